// Nearest-anchor projection of every key and value vector
// ("AnchorKV: Anchor-Residual KV Cache Compression", §3.1; anchors chosen per §3.2).
//
// Every vector x of a KV head is represented by the anchor a_j with the largest cosine
// similarity and the coefficient of the orthogonal projection onto span(a_j):
//   j* = argmax_j <x, a_j> / |a_j|   (|x| is common to all j and drops out)
//   gamma = <x, a_j*> / |a_j*|^2 = score_j* / |a_j*|
// Anchor positions represent themselves (slot = own, gamma = 1).
//
//   anchor_norm_kernel:  1 / |a| for every anchor row of K and V (0 for a zero row).
//   anchor_proj_kernel:  persistent; per (request, head, side, 128-token tile) unit the
//                        tile arrives by TMA, the anchors of (request, head, side) sit in
//                        shared memory in chunks of up to 256 rows, and one tcgen05 MMA
//                        chain per chunk writes the 128 x 256 dot products to TMEM.  Two
//                        sets of eight epilogue warps take alternate tiles (one TMEM
//                        accumulator each, four warps per column half) and keep the
//                        running arg-max per token.
#include <type_traits>

#include "internal.cuh"

namespace kvsel {
namespace {

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}


constexpr int kAnchorMax = 1024;       // anchors per (request, head) held in shared memory
constexpr int kAnChunk = 256;          // anchors per MMA chain (UMMA N)
constexpr int kApProducer = 16;        // warps 0-15: epilogue (eight per TMEM accumulator)
constexpr int kApMma = 17;
constexpr int kApThreads = 576;
constexpr int kApStages = 4;
constexpr int kApTile = 128 * 256;     // 128 tokens x 128 bf16: two K halves of 128 rows x 128 B
constexpr int kApB = kAnChunk * 256;   // 256 anchors x 128 bf16: two K halves of 256 rows x 128 B
constexpr size_t kApSmem = 1024 + static_cast<size_t>(kApStages) * kApTile + kApB + 2 * 2 * kAnchorMax * 4;

// the eight epilogue warps of accumulator p
__device__ __forceinline__ void eight_bar(int p) { asm volatile("bar.sync %0, 256;" ::"r"(1 + p) : "memory"); }

// One warp per anchor row: rows [0, rows) of K, then [0, rows) of V.
__global__ void __launch_bounds__(256) anchor_norm_kernel(const uint16_t* __restrict__ ak, const uint16_t* __restrict__ av,
                                                          long long rows, float* __restrict__ inv) {
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= 2 * rows) return;
  const uint16_t* src = w < rows ? ak + w * kHeadDim : av + (w - rows) * kHeadDim;
  const uint2 p = __ldg(reinterpret_cast<const uint2*>(src) + lane);
  const float x0 = __uint_as_float(p.x << 16), x1 = __uint_as_float(p.x & 0xFFFF0000u);
  const float x2 = __uint_as_float(p.y << 16), x3 = __uint_as_float(p.y & 0xFFFF0000u);
  float s = x0 * x0 + x1 * x1 + x2 * x2 + x3 * x3;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) inv[w] = s > 0.f ? 1.f / sqrtf(s) : 0.f;
}

struct Unit {
  int b, h, side, tile, seg, k, nch;
};

__device__ __forceinline__ Unit ap_unit(const AnchorArgs& a, int u) {
  Unit x;
  x.b = 0;
  while (x.b + 1 < a.rq.B && a.unit_base[x.b + 1] <= u) ++x.b;
  const int T = a.tiles[x.b];
  const int rem = u - a.unit_base[x.b];
  x.h = rem / (2 * T);
  const int r2 = rem - x.h * 2 * T;
  x.side = r2 / T;
  x.tile = r2 - x.side * T;
  x.seg = x.b * a.rq.H + x.h;
  const int c = __ldg(a.counts + x.seg);
  x.k = min(max(c, 0), kAnchorMax);
  x.nch = (x.k + kAnChunk - 1) / kAnChunk;
  return x;
}

__global__ void __launch_bounds__(kApThreads, 1)
    anchor_proj_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                       const __grid_constant__ CUtensorMap tak, const __grid_constant__ CUtensorMap tav,
                       const AnchorArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sA = smem;                                  // [stages][2 K halves][128 tokens][128 B]
  uint8_t* sB = smem + kApStages * kApTile;            // [2 K halves][256 anchors][128 B]
  float* s_inv = reinterpret_cast<float*>(sB + kApB);  // [2 groups][kAnchorMax]
  int* s_pos = reinterpret_cast<int*>(s_inv + 2 * kAnchorMax);

  __shared__ __align__(8) uint64_t afull[kApStages], aempty[kApStages], accf[2], acce[2];
  __shared__ __align__(8) uint64_t bfull, bempty, done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_mb[2][2][128];   // half merge: [accumulator][tile parity][token]
  __shared__ int s_mj[2][2][128];

  const int warp = warp_id(), lane = lane_id();
  int* status = a.wc.status;
  const int lo = static_cast<int>(static_cast<long long>(blockIdx.x) * a.units_total / gridDim.x);
  const int hi = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * a.units_total / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kApStages; ++s) {
      mbar_init(&afull[s], 1);
      mbar_init(&aempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&accf[s], 1);
      mbar_init(&acce[s], 8);
    }
    mbar_init(&bfull, 1);
    mbar_init(&bempty, 1);
    mbar_init(&done_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kApMma) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;

  if (warp == kApProducer) {
    if (lane == 0 && hi > lo) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tak);
      tma_prefetch_desc(&tav);
      long long prev_key = -1;
      int t = 0, bl = 0;
      bool ok = true;
      for (int u = lo; ok && u < hi; ++u) {
        const Unit x = ap_unit(a, u);
        if (x.nch == 0) continue;
        const int s = t % kApStages;
        if (!mbar_wait(&aempty[s], ((t / kApStages) & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&afull[s], kApTile);
        load_kv_tile(x.side ? &tv : &tk, a.src, x.b, x.h, a.rq.n[x.b], x.tile * 128, 128, sA + s * kApTile, &afull[s],
                     status);
        ++t;
        const long long base = __ldg(a.offsets + x.seg);
        for (int c = 0; c < x.nch; ++c) {
          const long long key = (static_cast<long long>(x.seg) * 2 + x.side) * 64 + c;
          if (key == prev_key) continue;
          if (bl > 0 && !mbar_wait(&bempty, (bl - 1) & 1, &s_abort, a.wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bfull, kApB);
          const int row0 = static_cast<int>(base) + c * kAnChunk;
          const CUtensorMap* m = x.side ? &tav : &tak;
          tma_load_2d(sB, m, &bfull, 0, row0);
          tma_load_2d(sB + kAnChunk * 128, m, &bfull, 64, row0);
          prev_key = key;
          ++bl;
        }
      }
      // drain copies still in flight
      for (int tt = max(0, t - kApStages); tt < t; ++tt) mbar_drain(&afull[tt % kApStages], (tt / kApStages) & 1, status);
      if (bl > 0) mbar_drain(&bfull, (bl - 1) & 1, status);
      ring_tail(aempty, kApStages, t, &s_abort, a.wc);
    }
  } else if (warp == kApMma) {
    if (lane == 0 && hi > lo) {
      long long prev_key = -1;
      int t = 0, bl = 0, ua0 = 0, ua1 = 0;   // uses of accumulator 0 / 1
      bool ok = true;
      const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(sB));
      for (int u = lo; ok && u < hi; ++u) {
        const Unit x = ap_unit(a, u);
        if (x.nch == 0) continue;
        const int acc = (u - lo) & 1;
        const int s = t % kApStages;
        if (!mbar_wait(&afull[s], (t / kApStages) & 1, &s_abort, a.wc)) break;
        const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + s * kApTile));
        for (int c = 0; c < x.nch; ++c) {
          const long long key = (static_cast<long long>(x.seg) * 2 + x.side) * 64 + c;
          if (key != prev_key) {
            if (bl > 0) umma_commit(&bempty);   // every MMA on the previous anchors is issued
            if (!mbar_wait(&bfull, bl & 1, &s_abort, a.wc)) {
              ok = false;
              break;
            }
            prev_key = key;
            ++bl;
          }
          if (!mbar_wait(&acce[acc], ((acc ? ua1 : ua0) & 1) ^ 1, &s_abort, a.wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nv = min(kAnChunk, x.k - c * kAnChunk);
          const uint32_t idesc = idesc_bf16_f32(128, (nv + 15) & ~15);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ao = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
            const uint32_t bo = ((kk >> 2) * (kAnChunk * 128) + (kk & 3) * 32) >> 4;
            umma_bf16(tbase + acc * 256, adesc + ao, bdesc + bo, idesc, kk ? 1u : 0u);
          }
          umma_commit(&accf[acc]);
          if (acc) ++ua1; else ++ua0;
        }
        umma_commit(&aempty[s]);   // the tile is read once the chain above completes
        ++t;
      }
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, status);
    }
  } else {
    // epilogue: warps 8p .. 8p+7 take the CTA's tiles of parity p (TMEM accumulator p);
    // `half` selects the columns [128 half, 128 half + 128) of each 256-anchor chunk and
    // q4 the TMEM lanes (tokens) [32 q4, 32 q4 + 32)
    const int p = warp >> 3, half = (warp >> 2) & 1, q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int pt = (warp & 7) * 32 + lane;   // thread index within the eight warps
    float* inv_p = s_inv + p * kAnchorMax;
    int* pos_p = s_pos + p * kAnchorMax;
    int ua = 0, par = 0;
    long long cur = -1;
    bool ok = true;
    for (int u = lo + p; u < hi; u += 2) {
      const Unit x = ap_unit(a, u);
      const long long key = static_cast<long long>(x.seg) * 2 + x.side;
      if (key != cur) {
        // anchors of (request, head, side): inverse norms and positions
        const long long base = __ldg(a.offsets + x.seg);
        eight_bar(p);
        for (int j = pt; j < x.k; j += 256) {
          const long long e = base + j;
          const bool in = e >= 0 && e < a.n_rows;
          inv_p[j] = in ? __ldg(a.inv + x.side * a.n_rows + e) : 0.f;
          pos_p[j] = in ? __ldg(a.idx + e) : -1;
        }
        eight_bar(p);
        cur = key;
      }
      const int tok = x.tile * 128 + r;
      // Arg-max by keyed maxima: within a 32-column round the score's five lowest mantissa
      // bits are replaced by 31 - (column in the round), so one float max per column
      // (three-input, over four independent partial maxima) finds the best score and,
      // among scores equal to 2^-18 relative, the lowest column.  Rounds are compared by
      // key (the earlier round on equal keys).  The decision and gamma carry that 2^-18
      // relative truncation of the score.
      float best = -INFINITY;
      int bround = 0;
      auto scan = [&](const float* y, int j0, int lim, auto full) {
        constexpr bool kFull = decltype(full)::value;
        float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < 32; q += 8) {
          const float4 i0 = *reinterpret_cast<const float4*>(inv_p + j0 + q);
          const float4 i1 = *reinterpret_cast<const float4*>(inv_p + j0 + q + 4);
          const float iv[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
          float kk[8];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            float sc0, sc1;   // the products two at a time (mul.rn.f32x2: the same rounding)
            unpack2(fmul2(pack2(y[q + e], y[q + e + 1]), pack2(iv[e], iv[e + 1])), sc0, sc1);
            kk[e] = __int_as_float((__float_as_int(sc0) & ~31) | (31 - (q + e)));
            kk[e + 1] = __int_as_float((__float_as_int(sc1) & ~31) | (31 - (q + e + 1)));
            if (!kFull && q + e >= lim) kk[e] = -INFINITY;
            if (!kFull && q + e + 1 >= lim) kk[e + 1] = -INFINITY;
          }
          m[(q >> 3) & 3] = fmax3(m[(q >> 3) & 3], fmax3(kk[0], kk[1], kk[2]), fmax3(kk[3], kk[4], kk[5]));
          m[((q >> 3) + 2) & 3] = fmax3(m[((q >> 3) + 2) & 3], kk[6], kk[7]);
        }
        const float mr = fmax3(m[0], m[1], fmaxf(m[2], m[3]));
        const bool gt = mr > best;
        bround = gt ? j0 : bround;
        best = gt ? mr : best;
      };
      for (int c = 0; c < x.nch; ++c) {
        ok = __all_sync(0xffffffffu, ok && mbar_wait(&accf[p], ua & 1, &s_abort, a.wc));
        const int nv = min(kAnChunk, x.k - c * kAnChunk) - half * 128;   // valid columns of this half
        if (ok && nv > 0) {
          tc_fence_after();
          const uint32_t taddr = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + p * 256 + half * 128;
          const int j0 = c * kAnChunk + half * 128;
          // 32-column rounds: TMEM load, wait, scan
          for (int c0 = 0; c0 < nv && c0 < 128; c0 += 32) {
            float y[32];
            tmem_ld32(taddr + c0, y);
            tmem_ld_wait();
            if (nv - c0 >= 32) scan(y, j0 + c0, 32, std::true_type{});
            else scan(y, j0 + c0, nv - c0, std::false_type{});
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[p]);
        ++ua;
      }
      // this half's best column, then the merge of the two halves (double-buffered by the
      // parity of the tile within the eight warps): larger truncated score, then lower column
      const int bj = best == -INFINITY ? 0 : bround + 31 - (__float_as_int(best) & 31);
      const float bq = __int_as_float(__float_as_int(best) & ~31);
      if (half == 1) {
        s_mb[p][par][r] = bq;
        s_mj[p][par][r] = bj;
      }
      // anchor positions represent themselves: binary search of the ascending list
      int self = -1;
      if (half == 0) {
        int l = 0, h2 = x.k;
        while (l < h2) {
          const int m = (l + h2) >> 1;
          if (pos_p[m] < tok) l = m + 1; else h2 = m;
        }
        if (l < x.k && pos_p[l] == tok) self = l;
      }
      eight_bar(p);
      if (half == 0) {
        float fb = bq;
        int fj = bj;
        const float ob = s_mb[p][par][r];
        const int oj = s_mj[p][par][r];
        if (ob > fb || (ob == fb && oj < fj)) {
          fb = ob;
          fj = oj;
        }
        const int n = a.rq.n[x.b];
        if (ok && tok < n) {
          const int slot = self >= 0 ? self : fj;
          const float gamma = self >= 0 ? 1.f : (x.k > 0 ? fb * inv_p[fj] : 0.f);
          const size_t o = a.rq.soff[x.b] + static_cast<size_t>(x.h) * n + tok;
          (x.side ? a.slot[1] : a.slot[0])[o] = slot;
          (x.side ? a.gamma[1] : a.gamma[0])[o] = gamma;
        }
      }
      par ^= 1;
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kApMma) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

int anchor_max() { return kAnchorMax; }

cudaError_t launch_anchor_norms(const uint16_t* ak, const uint16_t* av, long long rows, float* inv, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const long long threads = 2 * rows * 32;
  const int grid = static_cast<int>((threads + 255) / 256);
  anchor_norm_kernel<<<grid, 256, 0, st>>>(ak, av, rows, inv);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_anchor_project(const AnchorArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const CUtensorMap& tak, const CUtensorMap& tav, cudaStream_t st) {
  if (a.units_total <= 0) return cudaSuccess;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(anchor_proj_kernel), kApSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.units_total < sms ? a.units_total : sms;
  anchor_proj_kernel<<<grid, kApThreads, kApSmem, st>>>(tk, tv, tak, tav, a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
