// Query-agnostic scoring on tcgen05 tensor cores ("KVzip: Query-Agnostic KV Cache
// Compression with Context Reconstruction", §3.2: each key's importance is its maximum
// softmax weight over all queries and group heads; §3.4: queries are processed in chunks
// and the per-chunk maxima combined — max is associative, so the chunk size only bounds
// memory and does not change the result).
//
// Per KV head the queries are the G*n rows of Q[h] (all positions of all group heads),
// non-causal over all n keys:  S_i = max_r exp(l_ri - c_r),  c_r = log sum_j exp(l_rj).
//
//   qa_rowlse_kernel: A = a block of 512 query rows (4 M tiles), B = 128-key tiles
//     streamed over all n keys; every epilogue thread keeps an online (max, sum) for its
//     rows; writes c2_r = (m_r + log2 Z_r) in log2 units.
//   qa_keymax_kernel: A = a block of 256 keys (2 M tiles, resident), B = 256-row query
//     tiles streamed over a slice of the rows; every thread keeps max_r (l_ri*s2 - c2_r)
//     for its keys; slices merge with an order-preserving atomicMax in global memory.
//   qa_finish_kernel: s_raw_i = exp2(max).
// The softmax-free variant (KVzip §6.5, "KVzip-logit") skips the first pass: c2 = 0 and
// s2 = the logit scale, so the second pass keeps max_r l_ri itself and s_raw is that max.
// Both passes are tensor-core bound at this shape (2*G*n*n*d flop each).
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr float kNegBig = -1.0e30f;
constexpr int kMT = 4;                        // 128-row M tiles per CTA (512 rows or keys), resident
constexpr int kBlockHalf = kMT * 128 * 128;   // bytes of one column half of the resident block
constexpr int kNT = 128;                      // rows per streamed tile (keys in pass 1, queries in pass 2)
constexpr int kStages = 3;
constexpr int kTile = kNT * 256;              // bytes of one streamed tile (two 64-column halves)
constexpr uint32_t kSlotCols = kNT;           // one 128-column accumulator slot per M tile
constexpr uint32_t kTmemCols = kMT * kSlotCols;
// 16 epilogue warps (four per TMEM lane quadrant, 32 accumulator columns each), so that
// the latency of one warp's TMEM loads hides behind the others' arithmetic
constexpr int kEpiWarps = 16;
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 576;

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

__device__ __forceinline__ uint32_t f2key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Pass 1 streams 128-key tiles against 512 resident query rows: every UMMA is 128 x 128 x 16
// (N = 64 leaves the tensor pipe idle between short instructions) and the pass is paced by
// its exponentials.  Each M tile owns one 128-column TMEM accumulator; the epilogue
// releases it as soon as its columns are in registers, so the next tile's UMMAs for that M
// tile start while the other three are still being drained.

// ------------------------------------------------------------------------------------
// pass 1: log-sum-exp of every query row over all keys
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    qa_rowlse_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const QaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sQ = smem;                      // [4 M tiles][2 halves][128 rows][128 B]
  uint8_t* sK = smem + 2 * kBlockHalf;     // [stages][2 halves][128 keys][128 B]

  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], accf_bar[kMT], acce_bar[kMT];
  __shared__ __align__(8) uint64_t q_bar, done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = warp_id(), lane = lane_id();
  const int h = blockIdx.x / a.row_blocks;
  const int row0 = (blockIdx.x % a.row_blocks) * kMT * 128;
  const int n = a.n, GN = a.GN;
  const int ntiles = (n + kNT - 1) / kNT;
  int* status = a.wc.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < kMT; ++s) {
      mbar_init(&accf_bar[s], 1);
      mbar_init(&acce_bar[s], kEpiWarps);
    }
    mbar_init(&q_bar, 1);
    mbar_init(&done_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      mbar_arrive_expect_tx(&q_bar, 2 * kBlockHalf);
      const int qrow0 = h * GN + row0;
      for (int mt = 0; mt < kMT; ++mt)
        for (int rb = 0; rb < 128; rb += 64) {
          tma_load_2d(sQ + mt * 32768 + rb * 128, &tq, &q_bar, 0, qrow0 + mt * 128 + rb);
          tma_load_2d(sQ + mt * 32768 + 16384 + rb * 128, &tq, &q_bar, 64, qrow0 + mt * 128 + rb);
        }
      int t = 0;
      for (; t < ntiles; ++t) {
        const int s = t % kStages, u = t / kStages;
        if (!mbar_wait(&empty_bar[s], (u & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&full_bar[s], kTile);
        tma_load_4d(sK + s * kTile, &tk, &full_bar[s], 0, t * kNT, h, 0);
        tma_load_4d(sK + s * kTile + kNT * 128, &tk, &full_bar[s], 64, t * kNT, h, 0);
      }
      for (int tt = max(0, t - kStages); tt < t; ++tt) mbar_drain(&full_bar[tt % kStages], (tt / kStages) & 1, status);
      mbar_drain(&q_bar, 0, status);
      ring_tail(empty_bar, kStages, t, &s_abort, a.wc);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      bool ok = mbar_wait(&q_bar, 0, &s_abort, a.wc);
      constexpr uint32_t idesc = idesc_bf16_f32(128, kNT);
      const uint64_t qd0 = sdesc_kmajor_sw128(smem_u32(sQ));
      for (int t = 0; ok && t < ntiles; ++t) {
        const int s = t % kStages, u = t / kStages;
        if (!mbar_wait(&full_bar[s], u & 1, &s_abort, a.wc)) break;
        tc_fence_after();
        const uint64_t kd0 = sdesc_kmajor_sw128(smem_u32(sK + s * kTile));
#pragma unroll 1
        for (int mt = 0; mt < kMT; ++mt) {
          if (!mbar_wait(&acce_bar[mt], (t & 1) ^ 1, &s_abort, a.wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t koff = (k & 3) * 32;
            const uint64_t da = qd0 + ((mt * 32768 + (k >> 2) * 16384 + koff) >> 4);
            const uint64_t db = kd0 + (((k >> 2) * (kNT * 128) + koff) >> 4);
            umma_bf16(tbase + mt * kSlotCols, da, db, idesc, k > 0 ? 1u : 0u);
          }
          umma_commit(&accf_bar[mt]);
        }
        if (!ok) break;
        umma_commit(&empty_bar[s]);
      }
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, status);
    }
  } else {
    // thread = query row q4*32 + lane of every M tile; warp group cg takes keys [32cg, 32cg + 32)
    const int q4 = warp & 3, cg = warp >> 2;
    const float s2 = a.s2;
    float m[kMT], z[kMT];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      m[mt] = kNegBig;
      z[mt] = 0.f;
    }
    bool alive = true;
    for (int t = 0; alive && t < ntiles; ++t) {
      const int kc0 = t * kNT + cg * 32;
      const bool tail = kc0 + 32 > n;
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        bool ok = mbar_wait(&accf_bar[mt], t & 1, &s_abort, a.wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          alive = false;
          break;
        }
        tc_fence_after();
        float v[32];
        tmem_ld32(tbase + (static_cast<uint32_t>(q4 * 32) << 16) + mt * kSlotCols + cg * 32, v);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[mt]);
        if (tail) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (kc0 + j >= n) v[j] = -INFINITY;
        }
        float cmax = fmax3(v[0], v[1], v[2]);
#pragma unroll
        for (int j = 3; j < 31; j += 2) cmax = fmax3(cmax, v[j], v[j + 1]);
        cmax = fmaxf(cmax, v[31]);
        const float mn = fmaxf(m[mt], cmax * s2);
        // exp2(l * s2 - mn): packed FMA, four partial sums
        const uint64_t s2p = pack2(s2, s2), nmn = pack2(-mn, -mn);
        uint64_t p2[2] = {0ull, 0ull};
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float x0, x1, x2, x3;
          unpack2(ffma2(pack2(v[j + 0], v[j + 1]), s2p, nmn), x0, x1);
          unpack2(ffma2(pack2(v[j + 2], v[j + 3]), s2p, nmn), x2, x3);
          p2[0] = fadd2(p2[0], pack2(ex2_approx(x0), ex2_approx(x1)));
          p2[1] = fadd2(p2[1], pack2(ex2_approx(x2), ex2_approx(x3)));
        }
        float q0, q1;
        unpack2(fadd2(p2[0], p2[1]), q0, q1);
        z[mt] = z[mt] * ex2_approx(m[mt] - mn) + (q0 + q1);
        m[mt] = mn;
      }
    }
    // every UMMA has completed, so the streamed-tile buffers hold the key groups' partials
    float* s_xm = reinterpret_cast<float*>(sK);   // [3 key groups][kMT][4][32]
    float* s_xz = s_xm + 3 * kMT * 128;
    if (cg > 0) {
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        s_xm[(((cg - 1) * kMT + mt) * 4 + q4) * 32 + lane] = m[mt];
        s_xz[(((cg - 1) * kMT + mt) * 4 + q4) * 32 + lane] = z[mt];
      }
    }
    epi_bar();
    if (cg == 0 && alive) {
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const int r = row0 + mt * 128 + q4 * 32 + lane;
        float mm = m[mt];
#pragma unroll
        for (int g = 0; g < 3; ++g) mm = fmaxf(mm, s_xm[((g * kMT + mt) * 4 + q4) * 32 + lane]);
        float zz = z[mt] * ex2_approx(m[mt] - mm);
#pragma unroll
        for (int g = 0; g < 3; ++g) {
          const int i = ((g * kMT + mt) * 4 + q4) * 32 + lane;
          zz += s_xz[i] * ex2_approx(s_xm[i] - mm);
        }
        if (r < GN) a.c2[static_cast<size_t>(h) * GN + r] = mm + lg2_approx(zz);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// ------------------------------------------------------------------------------------
// pass 2: per key, max over a slice of query rows of (l * s2 - c2_row)
// ------------------------------------------------------------------------------------
// This pass has no exponentials, so it runs at the tensor pipe's pace, and 128 x 256 x 16
// UMMAs keep that pipe busier than N = 128: the resident block is 256 keys (two M tiles,
// one 256-column accumulator slot each) and query rows stream as 256-row tiles.
constexpr int kMT2 = 2;                       // resident 128-key M tiles
constexpr int kNT2 = 256;                     // query rows per streamed tile (UMMA N)
constexpr int kStages2 = 2;
constexpr int kKBlock2 = kMT2 * 32768;        // bytes of the resident keys
constexpr int kTile2 = kNT2 * 256;            // bytes of one streamed tile (two 64-column halves)
constexpr uint32_t kSlotCols2 = kNT2;         // one 256-column accumulator slot per M tile
constexpr int kRowsPerWarp2 = kNT2 / 4;       // query rows (accumulator columns) per epilogue warp
constexpr uint32_t kTmemCols2 = kMT2 * kSlotCols2;
static_assert(kTmemCols2 <= 512, "TMEM");

__global__ void __launch_bounds__(kThreads, 1)
    qa_keymax_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const QaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sK = smem;                      // [2 M tiles][2 halves][128 keys][128 B]
  uint8_t* sQ = smem + kKBlock2;           // [stages][2 halves][256 rows][128 B]

  __shared__ __align__(8) uint64_t full_bar[kStages2], empty_bar[kStages2], accf_bar[kMT2], acce_bar[kMT2];
  __shared__ __align__(8) uint64_t k_bar, done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(16) float s_nc[kEpiWarps][kRowsPerWarp2];   // -c2 of each warp's rows

  const int warp = warp_id(), lane = lane_id();
  const int per_head = a.key_blocks * a.row_splits;
  const int h = blockIdx.x / per_head;
  const int rem = blockIdx.x % per_head;
  const int kb = rem / a.row_splits, rs = rem % a.row_splits;
  const int key0 = kb * kMT2 * 128;
  const int n = a.n, GN = a.GN;
  // slices are whole tiles, so a tile never straddles two slices
  const int rows_per = ((GN + a.row_splits - 1) / a.row_splits + kNT2 - 1) / kNT2 * kNT2;
  const int r_begin = min(GN, rs * rows_per), r_end = min(GN, r_begin + rows_per);
  const int ntiles = r_end > r_begin ? (r_end - r_begin + kNT2 - 1) / kNT2 : 0;
  int* status = a.wc.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages2; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < kMT2; ++s) {
      mbar_init(&accf_bar[s], 1);
      mbar_init(&acce_bar[s], kEpiWarps);
    }
    mbar_init(&k_bar, 1);
    mbar_init(&done_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, kTmemCols2);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;

  if (warp == kProducerWarp) {
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      mbar_arrive_expect_tx(&k_bar, kKBlock2);
      for (int mt = 0; mt < kMT2; ++mt) {
        tma_load_4d(sK + mt * 32768, &tk, &k_bar, 0, key0 + mt * 128, h, 0);
        tma_load_4d(sK + mt * 32768 + 16384, &tk, &k_bar, 64, key0 + mt * 128, h, 0);
      }
      int t = 0;
      for (; t < ntiles; ++t) {
        const int s = t % kStages2, u = t / kStages2;
        if (!mbar_wait(&empty_bar[s], (u & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&full_bar[s], kTile2);
        const int qrow = h * GN + r_begin + t * kNT2;
        // the tensor map's box is 256 rows x 64 columns: one load per column half
        tma_load_2d(sQ + s * kTile2, &tq, &full_bar[s], 0, qrow);
        tma_load_2d(sQ + s * kTile2 + kNT2 * 128, &tq, &full_bar[s], 64, qrow);
      }
      for (int tt = max(0, t - kStages2); tt < t; ++tt) mbar_drain(&full_bar[tt % kStages2], (tt / kStages2) & 1, status);
      mbar_drain(&k_bar, 0, status);
      ring_tail(empty_bar, kStages2, t, &s_abort, a.wc);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && ntiles > 0) {
      bool ok = mbar_wait(&k_bar, 0, &s_abort, a.wc);
      constexpr uint32_t idesc = idesc_bf16_f32(128, kNT2);
      const uint64_t kd0 = sdesc_kmajor_sw128(smem_u32(sK));
      for (int t = 0; ok && t < ntiles; ++t) {
        const int s = t % kStages2, u = t / kStages2;
        if (!mbar_wait(&full_bar[s], u & 1, &s_abort, a.wc)) break;
        tc_fence_after();
        const uint64_t qd0 = sdesc_kmajor_sw128(smem_u32(sQ + s * kTile2));
#pragma unroll 1
        for (int mt = 0; mt < kMT2; ++mt) {
          if (!mbar_wait(&acce_bar[mt], (t & 1) ^ 1, &s_abort, a.wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t koff = (k & 3) * 32;
            const uint64_t da = kd0 + ((mt * 32768 + (k >> 2) * 16384 + koff) >> 4);
            const uint64_t db = qd0 + (((k >> 2) * (kNT2 * 128) + koff) >> 4);
            umma_bf16(tbase + mt * kSlotCols2, da, db, idesc, k > 0 ? 1u : 0u);
          }
          umma_commit(&accf_bar[mt]);
        }
        if (!ok) break;
        umma_commit(&empty_bar[s]);
      }
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, status);
    }
  } else {
    // thread = key q4*32 + lane of both M tiles; warp group cg takes query rows [64cg, 64cg + 64)
    const int q4 = warp & 3, cg = warp >> 2;
    const float s2 = a.s2;
    const float* c2h = a.c2 + static_cast<size_t>(h) * GN;
    float best[kMT2];
#pragma unroll
    for (int mt = 0; mt < kMT2; ++mt) best[mt] = -INFINITY;
    bool alive = true;
    // c2 of this warp's 64 rows, loaded a tile ahead (two rows per lane)
    auto load_c = [&](int t, int half) {
      const int rr = r_begin + t * kNT2 + cg * kRowsPerWarp2 + half * 32 + lane;
      return (t < ntiles && rr < r_end) ? (a.logit ? 0.f : __ldg(c2h + rr)) : INFINITY;
    };
    float cn0 = load_c(0, 0), cn1 = load_c(0, 1);
    const float4* nc4 = reinterpret_cast<const float4*>(&s_nc[warp][0]);
    for (int t = 0; alive && t < ntiles; ++t) {
      __syncwarp();   // the previous tile's reads of s_nc are done
      s_nc[warp][lane] = -cn0;
      s_nc[warp][32 + lane] = -cn1;
      __syncwarp();
      cn0 = load_c(t + 1, 0);
      cn1 = load_c(t + 1, 1);
#pragma unroll
      for (int mt = 0; mt < kMT2; ++mt) {
        bool ok = mbar_wait(&accf_bar[mt], t & 1, &s_abort, a.wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          alive = false;
          break;
        }
        tc_fence_after();
        float v[kRowsPerWarp2];
        const uint32_t taddr = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + mt * kSlotCols2 + cg * kRowsPerWarp2;
        tmem_ld32(taddr, v);
        tmem_ld32(taddr + 32, v + 32);
        tmem_ld_wait();
        // the columns are in registers: hand the slot back to the UMMA warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[mt]);
        float b0 = best[mt], b1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < kRowsPerWarp2; j += 4) {
          const float4 c = nc4[j >> 2];   // the same address in every lane: a broadcast
          b0 = fmax3(b0, fmaf(v[j], s2, c.x), fmaf(v[j + 1], s2, c.y));
          b1 = fmax3(b1, fmaf(v[j + 2], s2, c.z), fmaf(v[j + 3], s2, c.w));
        }
        best[mt] = fmaxf(b0, b1);
      }
    }
    // every UMMA has completed (each slot's last accumulator was waited for), so the
    // streamed-tile buffers are free to hold the row groups' partial maxima
    float* s_x = reinterpret_cast<float*>(sQ);   // [3 row groups][kMT2][4][32]
    if (cg > 0) {
#pragma unroll
      for (int mt = 0; mt < kMT2; ++mt) s_x[(((cg - 1) * kMT2 + mt) * 4 + q4) * 32 + lane] = best[mt];
    }
    epi_bar();
    if (cg == 0 && alive) {
#pragma unroll
      for (int mt = 0; mt < kMT2; ++mt) {
        const int key = key0 + mt * 128 + q4 * 32 + lane;
        float bm = best[mt];
#pragma unroll
        for (int g = 0; g < 3; ++g) bm = fmaxf(bm, s_x[((g * kMT2 + mt) * 4 + q4) * 32 + lane]);
        if (key < n && ntiles > 0) atomicMax(a.tmax + static_cast<size_t>(h) * n + key, f2key(bm));
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols2);
  }
}

__global__ void qa_finish_kernel(const uint32_t* __restrict__ tmax, float* __restrict__ s_raw, long long total,
                                 int logit) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float m = key2f(tmax[i]);
    s_raw[i] = logit ? m : ex2_approx(m);
  }
}

// One block per (request, head): maximum of the head's scores.
__global__ void head_max_kernel(const ReqTable rq, const float* __restrict__ s, float* __restrict__ out) {
  const int seg = blockIdx.x;
  const int b = seg / rq.H, h = seg - (seg / rq.H) * rq.H;
  const int n = rq.n[b];
  const float* src = s + rq.soff[b] + static_cast<long long>(h) * n;
  float m = -INFINITY;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, __ldg(src + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wm[32];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < blockDim.x / 32 ? wm[threadIdx.x] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) out[seg] = m;
  }
}

}  // namespace

cudaError_t launch_qa_rowlse(const QaArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t st) {
  const size_t smem = 1024 + 2 * kBlockHalf + kStages * kTile;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(qa_rowlse_kernel), smem);
  if (e != cudaSuccess) return e;
  qa_rowlse_kernel<<<a.H * a.row_blocks, kThreads, smem, st>>>(tq, tk, a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_qa_keymax(const QaArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t st) {
  const size_t smem = 1024 + kKBlock2 + kStages2 * kTile2;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(qa_keymax_kernel), smem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(a.tmax, 0, static_cast<size_t>(a.H) * a.n * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  qa_keymax_kernel<<<a.H * a.key_blocks * a.row_splits, kThreads, smem, st>>>(tq, tk, a);
  note_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long total = static_cast<long long>(a.H) * a.n;
  const int blocks = static_cast<int>((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  qa_finish_kernel<<<blocks, 256, 0, st>>>(a.tmax, a.s_raw, total, a.logit);
  note_launch();
  return cudaGetLastError();
}

int qa_block_rows() { return kMT * 128; }
int qa_key_block() { return kMT2 * 128; }
int qa_query_tile() { return kNT2; }

cudaError_t launch_head_max(const ReqTable& rq, const float* s, float* out, cudaStream_t st) {
  if (rq.B * rq.H <= 0) return cudaSuccess;
  head_max_kernel<<<rq.B * rq.H, 512, 0, st>>>(rq, s, out);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
