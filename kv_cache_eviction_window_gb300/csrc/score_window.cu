// Observation-window scoring on tcgen05 tensor cores
// ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", §3.4 Algorithm 2:
//  A = softmax(Q_hat K^T) over the last W queries, reduced over window rows; GQA: the
//  G query heads of a group share one KV head, "KVzip ...", §2.2).
//
// Exact softmax needs each row's max and normaliser over all n keys before any key's
// probability is final, so scoring runs in two passes over the key range:
//
//   pass 1 (win_rowstats_kernel): UMMA with A = window queries (M = 128 rows per tile),
//     B = a K tile (N keys), logits in TMEM; every epilogue thread owns one query row and
//     keeps an online (max, sum of exp) over its key chunk.  Partials per key chunk go
//     to the workspace.
//   pass 2 (win_keysum_kernel): UMMA with A = a K tile (M = 128 keys), B = all R window
//     rows; every epilogue thread owns one key and sums exp2(l*s2 - c_r) over the rows,
//     c_r = m_r + log2 Z_r merged from the pass-1 partials (or takes the max).
//
// Both passes stream K through a TMA ring (128-byte swizzled K-major tiles); K of a
// layer is re-read by pass 2 from L2 when nothing else ran in between.  Warp roles:
// warps 0-7 epilogue (two warps per TMEM lane quadrant: pass 1 splits a tile's columns
// between them, pass 2 gives each its own tiles when R <= 256), warp 8 TMA producer,
// warp 9 UMMA issuer.  Every wait is bounded (ptx.cuh).
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr float kNegBig = -1.0e30f;   // finite "minus infinity" for running maxima

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Barrier over the 8 epilogue warps that also ORs a predicate across them, so that an
// abort seen by one warp ends the loop of all of them at the same iteration.
__device__ __forceinline__ bool epi_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

// max of v[0..N): four independent chains of three-input max
template <int N>
__device__ __forceinline__ float tree_max(const float* v) {
  static_assert(N % 8 == 0, "N must be a multiple of 8");
  float t[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
  for (int j = 4; j < N - 4; j += 8) {
#pragma unroll
    for (int c = 0; c < 4; ++c) t[c] = fmax3(t[c], v[j + 2 * c], v[j + 2 * c + 1]);
  }
  // the loop above covers v[4 .. N-4); the last four values close the chains
  return fmax3(fmax3(t[0], t[1], v[N - 4]), fmax3(t[2], t[3], v[N - 3]), fmaxf(v[N - 2], v[N - 1]));
}

// sum of exp2(v[j] * s2 + c) over j < N: packed two-lane FMA and add, four accumulators
template <int N>
__device__ __forceinline__ float exp2_sum(const float* v, float s2, float mn) {
  static_assert(N % 8 == 0, "N must be a multiple of 8");
  const uint64_t s2p = pack2(s2, s2), nm = pack2(-mn, -mn);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    float x0, x1;
    unpack2(ffma2(pack2(v[j], v[j + 1]), s2p, nm), x0, x1);
    acc[(j >> 1) & 3] = fadd2(acc[(j >> 1) & 3], pack2(ex2_approx(x0), ex2_approx(x1)));
  }
  float a0, a1;
  unpack2(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), a0, a1);
  return a0 + a1;
}

__host__ __device__ constexpr uint32_t pow2_cols(uint32_t c) {
  return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512;
}

__device__ __forceinline__ void chunk_coords(const ChunkTable& ck, int B, int id, int& b, int& h, int& c) {
  b = 0;
  while (b + 1 < B && ck.base[b + 1] <= id) ++b;
  const int rem = id - ck.base[b];
  h = rem / ck.per_head[b];
  c = rem - h * ck.per_head[b];
}

// Window rows [0, R) of (b, h) from the 2-D query map (d, B*H*R rows), 32-row boxes,
// into [2 halves][R_pad rows][128 B].
__device__ __forceinline__ void load_q_rows(const CUtensorMap* map, int row0, int R, int half_bytes, uint8_t* dst,
                                            uint64_t* bar) {
  for (int rb = 0; rb < R; rb += 32) {
    tma_load_2d(dst + rb * 128, map, bar, 0, row0 + rb);
    tma_load_2d(dst + half_bytes + rb * 128, map, bar, 64, row0 + rb);
  }
}

// ------------------------------------------------------------------------------------
// pass 1: per-row max / sum of exp over one key chunk
// ------------------------------------------------------------------------------------
template <int MT, int NT, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    win_rowstats_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const WinScoreArgs a) {
  constexpr int kAcc = 2;
  constexpr uint32_t kAccCols = MT * NT;
  constexpr uint32_t kTmemCols = pow2_cols(kAcc * kAccCols);
  constexpr int kQHalf = MT * 128 * 128;
  constexpr int kKStage = NT * 256;
  constexpr int kCh = NT / 2;          // columns per epilogue thread per M tile
  static_assert(kCh % 32 == 0 && kCh <= 64, "column split");
  static_assert(kAcc * kAccCols <= 512, "TMEM");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + 2 * kQHalf;

  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], accf_bar[kAcc], acce_bar[kAcc];
  __shared__ __align__(8) uint64_t q_bar, done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_xm[MT][4][32], s_xz[MT][4][32];

  const int warp = warp_id(), lane = lane_id();
  int b, h, c;
  chunk_coords(a.ck, a.rq.B, blockIdx.x, b, h, c);
  const int n = a.rq.n[b];
  const int key_begin = c * a.ck.chunk_len;
  const int key_end = min(n, key_begin + a.ck.chunk_len);
  const int ntiles = key_end > key_begin ? (key_end - key_begin + NT - 1) / NT : 0;
  int* status = a.wc.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < kAcc; ++s) {
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
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      mbar_arrive_expect_tx(&q_bar, a.R * 256);
      load_q_rows(&tq, (b * a.rq.H + h) * a.R, a.R, kQHalf, sQ, &q_bar);
      int t = 0;
      for (; t < ntiles; ++t) {
        const int s = t % STAGES, u = t / STAGES;
        if (!mbar_wait(&empty_bar[s], (u & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&full_bar[s], kKStage);
        load_kv_tile(&tk, a.src, b, h, n, key_begin + t * NT, NT, sK + s * kKStage, &full_bar[s], status);
      }
      // every issued copy lands before the CTA can exit
      for (int tt = max(0, t - STAGES); tt < t; ++tt) mbar_drain(&full_bar[tt % STAGES], (tt / STAGES) & 1, status);
      mbar_drain(&q_bar, 0, status);
      ring_tail(empty_bar, STAGES, t, &s_abort, a.wc);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && ntiles > 0) {
      bool ok = mbar_wait(&q_bar, 0, &s_abort, a.wc);
      constexpr uint32_t idesc = idesc_bf16_f32(128, NT);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int s = t % STAGES, u = t / STAGES;
        const int acc = t % kAcc, ua = t / kAcc;
        if (!mbar_wait(&full_bar[s], u & 1, &s_abort, a.wc)) break;
        if (!mbar_wait(&acce_bar[acc], (ua & 1) ^ 1, &s_abort, a.wc)) break;
        tc_fence_after();
        // descriptors: the tile bases once, then byte offsets added to the address field
        const uint64_t kd0 = sdesc_kmajor_sw128(smem_u32(sK + s * kKStage));
        const uint64_t qd0 = sdesc_kmajor_sw128(smem_u32(sQ));
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t koff = (k & 3) * 32;
            const uint64_t da = qd0 + (((k >> 2) * kQHalf + mt * 16384 + koff) >> 4);
            const uint64_t db = kd0 + (((k >> 2) * (NT * 128) + koff) >> 4);
            umma_bf16(tbase + acc * kAccCols + mt * NT, da, db, idesc, k > 0 ? 1u : 0u);
          }
        }
        umma_commit(&empty_bar[s]);
        umma_commit(&accf_bar[acc]);
      }
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, status);
    }
  } else {
    // ---------------- epilogue: warps 0-7 ----------------
    const int q4 = warp & 3, cg = warp >> 2;
    const float s2 = a.s2;
    const int W = a.W, R = a.R;
    // keys below lim_all are visible to every row (causal bound of row w=0, and n)
    const int lim_all = a.causal ? (n - W + 1) : n;
    float m[MT], z[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      m[mt] = kNegBig;
      z[mt] = 0.f;
    }
    for (int t = 0; t < ntiles; ++t) {
      const int acc = t % kAcc, ua = t / kAcc;
      bool ok = mbar_wait(&accf_bar[acc], ua & 1, &s_abort, a.wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int kcol0 = key_begin + t * NT + cg * kCh;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        float v[kCh];
        const uint32_t taddr = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + acc * kAccCols + mt * NT + cg * kCh;
#pragma unroll
        for (int j = 0; j < kCh / 32; ++j) tmem_ld32(taddr + j * 32, v + j * 32);
        tmem_ld_wait();
        const int r = mt * 128 + q4 * 32 + lane;
        if (!(kcol0 + kCh <= lim_all) || r >= R) {
          const int lim_r = (r >= R) ? -1 : (a.causal ? min(n - 1, n - W + (r % W)) : n - 1);
#pragma unroll
          for (int j = 0; j < kCh; ++j)
            if (kcol0 + j > lim_r) v[j] = -INFINITY;
        }
        const float mn = fmaxf(m[mt], tree_max<kCh>(v) * s2);
        z[mt] = z[mt] * ex2_approx(m[mt] - mn) + exp2_sum<kCh>(v, s2, mn);
        m[mt] = mn;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar[acc]);
    }
    // merge the two column groups of each row and write the chunk partials
    if (cg == 1) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        s_xm[mt][q4][lane] = m[mt];
        s_xz[mt][q4][lane] = z[mt];
      }
    }
    epi_bar();
    if (cg == 0) {
      const int nch = a.ck.per_head[b], ncp = chunk_pad(nch);
      float* part = a.part + (static_cast<size_t>(a.ck.pbase[b]) + static_cast<size_t>(h) * ncp) * 2 * a.R_pad;
      float* pz = part + static_cast<size_t>(a.R_pad) * ncp;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int r = mt * 128 + q4 * 32 + lane;
        if (r < R) {
          const float m1 = s_xm[mt][q4][lane], z1 = s_xz[mt][q4][lane];
          const float mm = fmaxf(m[mt], m1);
          part[static_cast<size_t>(r) * ncp + c] = mm;
          pz[static_cast<size_t>(r) * ncp + c] = z[mt] * ex2_approx(m[mt] - mm) + z1 * ex2_approx(m1 - mm);
          if (c == nch - 1)   // neutral padding after the last chunk
            for (int j = nch; j < ncp; ++j) {
              part[static_cast<size_t>(r) * ncp + j] = kNegBig;
              pz[static_cast<size_t>(r) * ncp + j] = 0.f;
            }
        }
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
// pass 2: per-key sum (or max) of normalised window probabilities
// ------------------------------------------------------------------------------------
constexpr int kTileKeys = 128;
constexpr int kKTileBytes = kTileKeys * 256;

__global__ void __launch_bounds__(kThreads, 1)
    win_keysum_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const WinScoreArgs a, int stages, int nacc, uint32_t tmem_cols) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const int RP = a.R_pad;             // multiple of 64
  const int qhalf = RP * 128;
  uint8_t* sQ = smem;
  uint8_t* sK = smem + 2 * qhalf;
  float* s_c2 = reinterpret_cast<float*>(sK + stages * kKTileBytes);

  __shared__ __align__(8) uint64_t full_bar[4], empty_bar[4], accf_bar[4], acce_bar[4];
  __shared__ __align__(8) uint64_t q_bar, done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_x[4][32];

  const int warp = warp_id(), lane = lane_id();
  int b, h, c;
  chunk_coords(a.ck, a.rq.B, blockIdx.x, b, h, c);
  const int n = a.rq.n[b];
  const int key_begin = c * a.ck.chunk_len;
  const int key_end = min(n, key_begin + a.ck.chunk_len);
  const int ntiles = key_end > key_begin ? (key_end - key_begin + kTileKeys - 1) / kTileKeys : 0;
  int* status = a.wc.status;
  const int R = a.R;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < nacc; ++s) {
      mbar_init(&accf_bar[s], 1);
      // two or four accumulators: the four warps of one column group read each of them
      mbar_init(&acce_bar[s], nacc >= 2 ? 4 : kEpiWarps);
    }
    mbar_init(&q_bar, 1);
    mbar_init(&done_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, tmem_cols);
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
      mbar_arrive_expect_tx(&q_bar, R * 256);
      load_q_rows(&tq, (b * a.rq.H + h) * R, R, qhalf, sQ, &q_bar);
      int t = 0;
      for (; t < ntiles; ++t) {
        const int s = t % stages, u = t / stages;
        if (!mbar_wait(&empty_bar[s], (u & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&full_bar[s], kKTileBytes);
        load_kv_tile(&tk, a.src, b, h, n, key_begin + t * kTileKeys, kTileKeys, sK + s * kKTileBytes, &full_bar[s],
                     status);
      }
      for (int tt = max(0, t - stages); tt < t; ++tt) mbar_drain(&full_bar[tt % stages], (tt / stages) & 1, status);
      mbar_drain(&q_bar, 0, status);
      ring_tail(empty_bar, stages, t, &s_abort, a.wc);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && ntiles > 0) {
      bool ok = mbar_wait(&q_bar, 0, &s_abort, a.wc);
      for (int t = 0; ok && t < ntiles; ++t) {
        const int s = t % stages, u = t / stages;
        const int acc = t % nacc, ua = t / nacc;
        if (!mbar_wait(&full_bar[s], u & 1, &s_abort, a.wc)) break;
        if (!mbar_wait(&acce_bar[acc], (ua & 1) ^ 1, &s_abort, a.wc)) break;
        tc_fence_after();
        const uint64_t kd0 = sdesc_kmajor_sw128(smem_u32(sK + s * kKTileBytes));
        const uint64_t qd0 = sdesc_kmajor_sw128(smem_u32(sQ));
        for (int n0 = 0; n0 < R; n0 += 256) {
          const int nc = min(256, R - n0);
          const uint32_t idesc = idesc_bf16_f32(128, nc);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t koff = (k & 3) * 32;
            const uint64_t da = kd0 + (((k >> 2) * (kTileKeys * 128) + koff) >> 4);
            const uint64_t db = qd0 + (static_cast<uint32_t>((k >> 2) * qhalf + n0 * 128 + koff) >> 4);
            umma_bf16(tbase + acc * RP + n0, da, db, idesc, k > 0 ? 1u : 0u);
          }
        }
        umma_commit(&empty_bar[s]);
        umma_commit(&accf_bar[acc]);
      }
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, status);
    }
  } else {
    // ---------------- epilogue: warps 0-7 ----------------
    // merged row statistics c2[r] = m_r + log2 Z_r  (log2 units); a row's chunk
    // partials are contiguous, read as float4
    {
      const int ncp = chunk_pad(a.ck.per_head[b]);
      const float* pm = a.part + (static_cast<size_t>(a.ck.pbase[b]) + static_cast<size_t>(h) * ncp) * 2 * RP;
      const float* pz = pm + static_cast<size_t>(RP) * ncp;
      for (int r = threadIdx.x; r < RP; r += kEpiWarps * 32) {
        float c2 = 0.f;
        if (r < R) {
          const float4* m4 = reinterpret_cast<const float4*>(pm + static_cast<size_t>(r) * ncp);
          const float4* z4 = reinterpret_cast<const float4*>(pz + static_cast<size_t>(r) * ncp);
          float mm = kNegBig;
#pragma unroll 4
          for (int j = 0; j < ncp / 4; ++j) {
            const float4 v = m4[j];
            mm = fmaxf(mm, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
          }
          float zz = 0.f;
#pragma unroll 4
          for (int j = 0; j < ncp / 4; ++j) {
            const float4 v = m4[j], w = z4[j];
            zz += w.x * ex2_approx(v.x - mm) + w.y * ex2_approx(v.y - mm) + w.z * ex2_approx(v.z - mm) +
                  w.w * ex2_approx(v.w - mm);
          }
          c2 = mm + lg2_approx(zz);
        }
        s_c2[r] = -c2;   // stored negated: the epilogue adds it with a fused multiply-add
      }
    }
    epi_bar();
    const int q4 = warp & 3, cg = warp >> 2;
    const float s2 = a.s2;
    const int W = a.W;
    const bool is_max = (a.reduce == 2);
    const float row_scale = (a.reduce == 1) ? 1.f / static_cast<float>(R) : 1.f;
    const size_t out_base = static_cast<size_t>(a.rq.soff[b]) + static_cast<size_t>(h) * n;
    if (nacc >= 2) {
      // warp (q4, cg) takes tiles cg, cg + 2, ... (accumulators of parity cg) and sums
      // every window row of its key alone: no exchange between the warps of a tile.
      // Rows go in blocks of 32 (one TMEM load each, the next one issued before the
      // current block is summed); masked rows (causal tail, rows past R) become -inf.
      const uint64_t s2p = pack2(s2, s2);
      auto rows32 = [&](float (&v)[32], int ca, int wmin, float& acc_sum, float& acc_max) {
        if (wmin > 0 || ca + 32 > R) {
          int w = ca % W;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (ca + j >= R || w < wmin) v[j] = -INFINITY;
            w = (w + 1 == W) ? 0 : w + 1;
          }
        }
        const float4* nc4 = reinterpret_cast<const float4*>(s_c2 + ca);   // -c2 of rows ca ..
        if (is_max) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 c = nc4[j >> 2];
            acc_max = fmax3(acc_max, fmaf(v[j], s2, c.x), fmaf(v[j + 1], s2, c.y));
            acc_max = fmax3(acc_max, fmaf(v[j + 2], s2, c.z), fmaf(v[j + 3], s2, c.w));
          }
        } else {
          uint64_t p2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 c = nc4[j >> 2];
            float x0, x1, x2, x3;
            unpack2(ffma2(pack2(v[j], v[j + 1]), s2p, pack2(c.x, c.y)), x0, x1);
            unpack2(ffma2(pack2(v[j + 2], v[j + 3]), s2p, pack2(c.z, c.w)), x2, x3);
            p2[(j >> 2) & 3] = fadd2(p2[(j >> 2) & 3], pack2(ex2_approx(x0), ex2_approx(x1)));
            p2[(j >> 2) & 3] = fadd2(p2[(j >> 2) & 3], pack2(ex2_approx(x2), ex2_approx(x3)));
          }
          float q0, q1;
          unpack2(fadd2(fadd2(p2[0], p2[1]), fadd2(p2[2], p2[3])), q0, q1);
          acc_sum += q0 + q1;
        }
      };
      for (int t = cg; t < ntiles; t += 2) {
        const int acc = t % nacc, ua = t / nacc;
        const bool ok = mbar_wait(&accf_bar[acc], ua & 1, &s_abort, a.wc);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        const int key = key_begin + t * kTileKeys + q4 * 32 + lane;
        // causal: row r sees this key iff (r % W) >= key - (n - W)
        const int wmin = a.causal ? key - (n - W) : -1;
        float acc_sum = 0.f, acc_max = -INFINITY;
        const uint32_t trow = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + acc * RP;
        float va[32], vb[32];
        tmem_ld32(trow, va);
#pragma unroll 1
        for (int c0 = 0; c0 < R; c0 += 64) {
          tmem_ld_wait();   // rows c0 .. c0 + 31
          const bool second = c0 + 32 < R;
          if (second) tmem_ld32(trow + c0 + 32, vb);
          const bool last_a = !second;
          if (last_a) {   // every row of the tile is in registers: release the accumulator
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce_bar[acc]);
          }
          rows32(va, c0, wmin, acc_sum, acc_max);
          if (second) {
            tmem_ld_wait();   // rows c0 + 32 .. c0 + 63
            const bool more = c0 + 64 < R;
            if (more) {
              tmem_ld32(trow + c0 + 64, va);
            } else {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acce_bar[acc]);
            }
            rows32(vb, c0 + 32, wmin, acc_sum, acc_max);
          }
        }
        if (key < n) a.s_raw[out_base + key] = is_max ? ex2_approx(acc_max) : acc_sum * row_scale;
      }
    } else {
      // one accumulator (R > 256): both column groups read every tile, each half the rows
      const int half_cols = RP / 2;   // multiple of 32
      const int col0 = cg * half_cols;
      const int col_end = min(R, col0 + half_cols);
      for (int t = 0; t < ntiles; ++t) {
        const int acc = t % nacc, ua = t / nacc;
        const bool ok = mbar_wait(&accf_bar[acc], ua & 1, &s_abort, a.wc);
        if (epi_any(!ok)) break;
        tc_fence_after();
        const int key = key_begin + t * kTileKeys + q4 * 32 + lane;
        const int wmin = a.causal ? key - (n - W) : -1;
        float acc_sum = 0.f, acc_max = -INFINITY;
        const uint32_t trow = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + acc * RP;
        for (int c0 = col0; c0 < col_end; c0 += 64) {
          float v[64];
          const int cnt = min(64, col_end - c0);   // warp-uniform
          tmem_ld32(trow + c0, v);
          if (cnt > 32) tmem_ld32(trow + c0 + 32, v + 32);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int r = c0 + j;
            if (j < cnt && (r % W) >= wmin) {
              const float y = fmaf(v[j], s2, s_c2[r]);
              if (is_max)
                acc_max = fmaxf(acc_max, y);
              else
                acc_sum += ex2_approx(y);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[acc]);
        float part_v = is_max ? acc_max : acc_sum;
        if (cg == 1) s_x[q4][lane] = part_v;
        epi_bar();
        if (cg == 0 && key < n) {
          const float o = s_x[q4][lane];
          a.s_raw[out_base + key] = is_max ? ex2_approx(fmaxf(part_v, o)) : (part_v + o) * row_scale;
        }
        epi_bar();
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, tmem_cols);
  }
}

// ------------------------------------------------------------------------------------
// both passes in one cooperative launch (one key chunk per CTA, all CTAs co-resident)
// ------------------------------------------------------------------------------------
// Pass 1 as win_rowstats_kernel; then a bounded grid barrier (the row partials of every
// chunk of this (request, head) are written); then pass 2 over the CTA's own chunk, whose
// K tiles are still in L2.  The TMA producer and the UMMA warp run straight on into
// pass 2 (K and Q do not depend on the barrier); only the epilogue waits.
//
// Shared-memory matrix descriptor: K-major operand, 32-byte swizzle.  Rows are 32 B
// (16 bf16: one UMMA K step), 8-row groups (256 B) follow each other.  `saddr` must be
// 256-byte aligned.  The swizzle only exchanges the two 16-byte halves of a row, so an
// operand whose other side is constant along K may be written without it.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw32(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address      [0,14)
  d |= static_cast<uint64_t>(1u) << 16;                  // leading byte off.  [16,30)
  d |= static_cast<uint64_t>(256u >> 4) << 32;           // stride byte offset [32,46)
  d |= static_cast<uint64_t>(1u) << 46;                  // descriptor version [46,48)
  d |= static_cast<uint64_t>(6u) << 61;                  // swizzle: 32 B      [61,64)
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// The epilogue has 16 warps, four per TMEM lane quadrant, so that every SM sub-partition
// keeps four warps of exponentials in flight.  Pass 1: each warp takes a 32-key column
// group of every tile.  Pass 2: two groups of eight warps take alternate tiles; in a
// group the two warps of a lane quadrant split the window rows in halves and add their
// partial sums through shared memory.
//
// Pass 2 needs l_rj * s2 - c2_r for every window row r, c2_r = m_r + log2 Z_r.  The row
// constant is added by the tensor core, not the epilogue: one more K step multiplies a
// block of ones (keys side) by the constants -c2_r / s2 split into three bf16 parts
// (rows side), so the accumulator holds l_rj - c2_r / s2 and the epilogue only scales it.
// Reading 64 constants from shared memory per tile would queue behind the UMMA operand
// reads, which keep the shared-memory port busy during pass 2.
//
// Two warps issue the UMMAs, one the even tiles and one the odd ones (each with its own
// accumulators and commits).  One issuing thread spends about 54 cycles per M = 128,
// N = 128 UMMA and more per commit and wait, while the tensor core needs 64 cycles per
// such UMMA, so a single issuer leaves the tensor core idle for part of every tile.
constexpr int kFEpiWarps = 16;
constexpr int kFProducerWarp = 16;
constexpr int kFMmaWarp = 17;       // UMMA issue: warps 17 and 18 take alternate tiles
constexpr int kFThreads = 608;

__device__ __forceinline__ void fused_epi_bar() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

__device__ __forceinline__ bool fused_epi_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 512, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

// barrier over the 256 threads of pass-2 group `grp` that ANDs a predicate across them
__device__ __forceinline__ bool group_all(int grp, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(2 + grp)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void group_bar(int grp) { asm volatile("bar.sync %0, 256;" ::"r"(4 + grp) : "memory"); }

template <int MT>
__global__ void __launch_bounds__(kFThreads, 1)
    win_fused_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const WinScoreArgs a, unsigned int* grid_count) {
  constexpr int NT = 128, STAGES = (MT == 1) ? 5 : 4, kAcc = 2;
  // pass-2 accumulators: R <= 128 uses eight half-tile accumulators (N = R/2, columns
  // 128c and 128c + 64 for tile class c = t % 4); R > 128 uses two of N = R
  constexpr int kAcc2 = (MT == 1) ? 8 : 2;
  constexpr uint32_t kAccCols = MT * 128;
  constexpr uint32_t kTmemCols = 512;
  constexpr int kQHalf = MT * 128 * 128;
  constexpr int kKStage = NT * 256;
  constexpr int kCg = 32;                            // pass-1 keys per warp and tile

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + 2 * kQHalf;
  uint8_t* sOnes = sK + STAGES * kKStage;   // 128 rows x 16 bf16 ones (32-byte swizzle rows)
  uint8_t* sC = sOnes + 128 * 32;           // MT*128 rows x 16 bf16: -c2_r / s2 in three parts

  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t accf1[kAcc], acce1[kAcc], accf2[kAcc2], acce2[kAcc2];
  __shared__ __align__(8) uint64_t q_bar, done_bar[2], c_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_xm[MT][4][128], s_xz[MT][4][128];   // pass-1 partials per column group
  __shared__ float s_part[2][128];                         // pass-2 half sums per group

  const int warp = warp_id(), lane = lane_id();
  int b, h, c;
  chunk_coords(a.ck, a.rq.B, blockIdx.x, b, h, c);
  const int n = a.rq.n[b];
  const int key_begin = c * a.ck.chunk_len;
  const int key_end = min(n, key_begin + a.ck.chunk_len);
  const int ntiles = key_end > key_begin ? (key_end - key_begin + NT - 1) / NT : 0;
  int* status = a.wc.status;
  const int R = a.R, RP = a.R_pad;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < kAcc; ++s) {
      mbar_init(&accf1[s], 1);
      mbar_init(&acce1[s], kFEpiWarps);
    }
    for (int s = 0; s < kAcc2; ++s) {
      mbar_init(&accf2[s], 1);
      mbar_init(&acce2[s], MT == 1 ? 4 : kFEpiWarps / 2);   // the warps that read one pass-2 accumulator
    }
    mbar_init(&q_bar, 1);
    mbar_init(&done_bar[0], 1);
    mbar_init(&done_bar[1], 1);
    mbar_init(&c_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 128 * 32 / 16; i += kFThreads)   // bf16 1.0 = 0x3f80
    reinterpret_cast<uint4*>(sOnes)[i] = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
  fence_proxy_async_smem();
  if (warp == kFMmaWarp) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  if (a.nu_zero != nullptr && warp < kFEpiWarps) {   // this chunk's value norms start from zero
    float* z = a.nu_zero + static_cast<size_t>(a.rq.soff[b]) + static_cast<size_t>(h) * n;
    for (int k = key_begin + static_cast<int>(threadIdx.x); k < key_end; k += kFEpiWarps * 32) z[k] = 0.f;
  }

  if (warp == kFProducerWarp) {
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      mbar_arrive_expect_tx(&q_bar, R * 256);
      load_q_rows(&tq, (b * a.rq.H + h) * R, R, kQHalf, sQ, &q_bar);
      int T = 0;
      for (; T < 2 * ntiles; ++T) {   // pass 1 tiles, then the same tiles again for pass 2
        const int s = T % STAGES, u = T / STAGES;
        if (!mbar_wait(&empty_bar[s], (u & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&full_bar[s], kKStage);
        const int t = T < ntiles ? T : T - ntiles;
        load_kv_tile(&tk, a.src, b, h, n, key_begin + t * NT, NT, sK + s * kKStage, &full_bar[s], status);
      }
      for (int tt = max(0, T - STAGES); tt < T; ++tt) mbar_drain(&full_bar[tt % STAGES], (tt / STAGES) & 1, status);
      mbar_drain(&q_bar, 0, status);
      ring_tail(empty_bar, STAGES, T, &s_abort, a.wc);
    }
  } else if (warp == kFMmaWarp || warp == kFMmaWarp + 1) {
    const int iss = warp - kFMmaWarp;   // this warp issues tiles iss, iss + 2, ...
    if (lane == 0 && ntiles > iss) {
      bool ok = mbar_wait(&q_bar, 0, &s_abort, a.wc);
      const uint64_t qd0 = sdesc_kmajor_sw128(smem_u32(sQ));
      // pass 1: A = window rows, B = keys (accumulator t % 2 = iss)
      constexpr uint32_t idesc1 = idesc_bf16_f32(128, NT);
      for (int t = iss; ok && t < ntiles; t += 2) {
        const int s = t % STAGES, u = t / STAGES;
        const int acc = t % kAcc, ua = t / kAcc;
        if (!mbar_wait(&full_bar[s], u & 1, &s_abort, a.wc) ||
            !mbar_wait(&acce1[acc], (ua & 1) ^ 1, &s_abort, a.wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kd0 = sdesc_kmajor_sw128(smem_u32(sK + s * kKStage));
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t koff = (k & 3) * 32;
            umma_bf16(tbase + acc * kAccCols + mt * NT, qd0 + (((k >> 2) * kQHalf + mt * 16384 + koff) >> 4),
                      kd0 + (((k >> 2) * (NT * 128) + koff) >> 4), idesc1, k > 0 ? 1u : 0u);
          }
        }
        umma_commit(&empty_bar[s]);
        umma_commit(&accf1[acc]);
      }
      // pass 2: A = keys (M = 128), B = window rows; a ninth K step adds -c2_r / s2
      // (ones x C).  The logits of the first tiles (as many as there are accumulators) are
      // issued before the row statistics exist (during the grid barrier); their constants
      // follow.  A pass-2 tile's columns always belong to the pass-1 accumulator of the
      // same parity, so this warp reuses only columns it used in pass 1.
      const uint64_t onesd = sdesc_kmajor_sw32(smem_u32(sOnes));
      auto add_row_consts = [&](int acc) {
        for (int n0 = 0; n0 < R; n0 += 256) {
          const int nc = min(256, R - n0);
          umma_bf16(tbase + acc * kAccCols + n0, onesd, sdesc_kmajor_sw32(smem_u32(sC + n0 * 32)),
                    idesc_bf16_f32(128, nc), 1u);
        }
      };
      if constexpr (MT == 1) {
        // tile t (class c = t % 4) fills accumulator halves 2c (window rows [0, R/2)) and
        // 2c + 1 (rows [R/2, R)); the epilogue releases each half when it has summed it,
        // so the next tile of the class starts while the second half is being summed
        const int Rh = R / 2;
        const uint32_t idesc_h = idesc_bf16_f32(128, Rh);
        auto logits_half = [&](uint64_t kd0, int hcol, int r0) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t koff = (k & 3) * 32;
            umma_bf16(tbase + hcol, kd0 + (((k >> 2) * (NT * 128) + koff) >> 4),
                      qd0 + (static_cast<uint32_t>((k >> 2) * kQHalf + r0 * 128 + koff) >> 4), idesc_h,
                      k > 0 ? 1u : 0u);
          }
        };
        auto consts_half = [&](int hcol, int r0) {
          umma_bf16(tbase + hcol, onesd, sdesc_kmajor_sw32(smem_u32(sC + r0 * 32)), idesc_h, 1u);
        };
        const int early = min(ntiles, 4);
        for (int t = iss; ok && t < ntiles; t += 2) {
          const int T = ntiles + t;
          const int s = T % STAGES, u = T / STAGES;
          const int c = t & 3, uc = t >> 2;
          if (!mbar_wait(&full_bar[s], u & 1, &s_abort, a.wc)) {
            ok = false;
            break;
          }
          const uint64_t kd0 = sdesc_kmajor_sw128(smem_u32(sK + s * kKStage));
          for (int hh = 0; ok && hh < 2; ++hh) {
            const int ai = 2 * c + hh;
            if (t < 4) {
              // columns 128c .. 128c + 127 were pass-1 accumulator c: wait for its last release
              if (hh == 0 && c < kAcc) {
                const int last1 = ((ntiles - 1 - c) >= 0) ? ntiles - 1 - ((ntiles - 1 - c) % kAcc) : -1;
                if (last1 >= 0 && !mbar_wait(&acce1[c], (last1 / kAcc) & 1, &s_abort, a.wc)) ok = false;
              }
            } else if (!mbar_wait(&acce2[ai], (uc & 1) ^ 1, &s_abort, a.wc)) {
              ok = false;
            }
            if (!ok) break;
            tc_fence_after();
            logits_half(kd0, 128 * c + 64 * hh, hh * Rh);
            if (t >= early) {
              consts_half(128 * c + 64 * hh, hh * Rh);
              umma_commit(&accf2[ai]);
            }
          }
          if (!ok) break;
          umma_commit(&empty_bar[s]);   // the K stage is free once both halves' logits are done
          if (t < early && t + 2 >= early) {   // this warp's last tile issued before the constants
            if (!mbar_wait(&c_bar, 0, &s_abort, a.wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int t2 = iss; t2 <= t; t2 += 2)
              for (int hh = 0; hh < 2; ++hh) {
                consts_half(128 * (t2 & 3) + 64 * hh, hh * Rh);
                umma_commit(&accf2[2 * (t2 & 3) + hh]);
              }
          }
        }
      } else {
        const int early = min(ntiles, kAcc2);
        for (int t = iss; ok && t < ntiles; t += 2) {
          const int T = ntiles + t;
          const int s = T % STAGES, u = T / STAGES;
          const int acc = t % kAcc2, ua = t / kAcc2;
          if (!mbar_wait(&full_bar[s], u & 1, &s_abort, a.wc)) {
            ok = false;
            break;
          }
          if (t < kAcc2) {
            // first pass-2 use of these columns: pass 1's last use of them is released
            if (acc < kAcc) {
              const int last1 = ((ntiles - 1 - acc) >= 0) ? ntiles - 1 - ((ntiles - 1 - acc) % kAcc) : -1;
              if (last1 >= 0 && !mbar_wait(&acce1[acc], (last1 / kAcc) & 1, &s_abort, a.wc)) {
                ok = false;
                break;
              }
            }
          } else if (!mbar_wait(&acce2[acc], (ua & 1) ^ 1, &s_abort, a.wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd0 = sdesc_kmajor_sw128(smem_u32(sK + s * kKStage));
          for (int n0 = 0; n0 < R; n0 += 256) {
            const int nc = min(256, R - n0);
            const uint32_t idesc = idesc_bf16_f32(128, nc);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t koff = (k & 3) * 32;
              umma_bf16(tbase + acc * kAccCols + n0, kd0 + (((k >> 2) * (NT * 128) + koff) >> 4),
                        qd0 + (static_cast<uint32_t>((k >> 2) * kQHalf + n0 * 128 + koff) >> 4), idesc, k > 0 ? 1u : 0u);
            }
          }
          umma_commit(&empty_bar[s]);   // the K stage is free once the logits are done
          if (t < early && t + 2 >= early) {   // this warp's last tile issued before the constants
            if (!mbar_wait(&c_bar, 0, &s_abort, a.wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int t2 = iss; t2 <= t; t2 += 2) {
              add_row_consts(t2 % kAcc2);
              umma_commit(&accf2[t2 % kAcc2]);
            }
          } else if (t >= early) {
            add_row_consts(acc);
            umma_commit(&accf2[acc]);
          }
        }
      }
      umma_commit(&done_bar[iss]);
      mbar_drain(&done_bar[iss], 0, status);
    }
  } else {
    // ---------------- epilogue, pass 1: warp (q4, cg) takes keys [32cg, 32cg + 32) of a tile ----------------
    const int q4 = warp & 3, cg = warp >> 2;
    const float s2 = a.s2;
    const int W = a.W;
    const int lim_all = a.causal ? (n - W + 1) : n;
    float m[MT], z[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      m[mt] = kNegBig;
      z[mt] = 0.f;
    }
    bool alive = true;
    for (int t = 0; t < ntiles; ++t) {
      const int acc = t % kAcc, ua = t / kAcc;
      bool ok = mbar_wait(&accf1[acc], ua & 1, &s_abort, a.wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        alive = false;
        break;
      }
      tc_fence_after();
      float v[MT][kCg];
      const uint32_t taddr = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + acc * kAccCols + cg * kCg;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) tmem_ld32(taddr + mt * NT, v[mt]);
      tmem_ld_wait();
      // the logits are in registers: hand the accumulator back to the UMMA warp now
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce1[acc]);
      const int kcol0 = key_begin + t * NT + cg * kCg;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int r = mt * 128 + q4 * 32 + lane;
        if (!(kcol0 + kCg <= lim_all) || r >= R) {
          const int lim_r = (r >= R) ? -1 : (a.causal ? min(n - 1, n - W + (r % W)) : n - 1);
#pragma unroll
          for (int j = 0; j < kCg; ++j)
            if (kcol0 + j > lim_r) v[mt][j] = -INFINITY;
        }
        const float mn = fmaxf(m[mt], tree_max<kCg>(v[mt]) * s2);
        z[mt] = z[mt] * ex2_approx(m[mt] - mn) + exp2_sum<kCg>(v[mt], s2, mn);
        m[mt] = mn;
      }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      s_xm[mt][cg][q4 * 32 + lane] = m[mt];
      s_xz[mt][cg][q4 * 32 + lane] = z[mt];
    }
    fused_epi_bar();
    const int nch = a.ck.per_head[b], ncp = chunk_pad(nch);
    float* pm = a.part + (static_cast<size_t>(a.ck.pbase[b]) + static_cast<size_t>(h) * ncp) * 2 * RP;
    float* pz = pm + static_cast<size_t>(RP) * ncp;
    if (cg == 0) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int rl = q4 * 32 + lane, r = mt * 128 + rl;
        if (r < R) {
          float mm = s_xm[mt][0][rl];
#pragma unroll
          for (int g = 1; g < 4; ++g) mm = fmaxf(mm, s_xm[mt][g][rl]);
          float zz = 0.f;
#pragma unroll
          for (int g = 0; g < 4; ++g) zz += s_xz[mt][g][rl] * ex2_approx(s_xm[mt][g][rl] - mm);
          pm[static_cast<size_t>(r) * ncp + c] = mm;
          pz[static_cast<size_t>(r) * ncp + c] = zz;
          if (c == nch - 1)
            for (int j = nch; j < ncp; ++j) {
              pm[static_cast<size_t>(r) * ncp + j] = kNegBig;
              pz[static_cast<size_t>(r) * ncp + j] = 0.f;
            }
        }
      }
    }
    // ---------------- grid barrier: every chunk's partials are in memory ----------------
    fused_epi_bar();
    if (threadIdx.x == 0) {
      // only the chunks of this (request, head) are needed: an arrival and a departure
      // count per head.  Every CTA arrives and departs exactly once (also after a timeout),
      // and the last to depart zeroes both, so the counters are ready for the next launch
      // without a memset.
      unsigned int* arrive = grid_count + 2 * (b * a.rq.H + h);
      unsigned int* depart = arrive + 1;
      __threadfence();
      atomicAdd(arrive, 1u);
      const long long t0 = clock64();
      while (true) {
        const unsigned int v = *reinterpret_cast<volatile unsigned int*>(arrive);
        if (v >= static_cast<unsigned int>(nch)) break;
        if (*reinterpret_cast<volatile int*>(&s_abort) ||
            static_cast<unsigned long long>(clock64() - t0) > a.wc.limit) {
          s_abort = 1;
          atomicOr(status, DEV_TIMEOUT_PIPE);
          break;
        }
      }
      __threadfence();
      if (atomicAdd(depart, 1u) == static_cast<unsigned int>(nch) - 1u) {
        atomicExch(arrive, 0u);
        atomicExch(depart, 0u);
      }
    }
    if (fused_epi_any(!alive || *reinterpret_cast<volatile int*>(&s_abort) != 0)) alive = false;
    if (alive) {
      // merged row statistics c2[r] = m_r + log2 Z_r (log2 units): kTpr threads per row
      // split its chunk partials (float4 groups, all loads issued first), then combine
      {
        constexpr int kTpr = (kFEpiWarps * 32) / (MT * 128);   // 4 (R <= 128) or 2
        constexpr int kMaxG = 64 / 4 / kTpr;                   // float4 groups per thread (ncp <= 64)
        const int r = threadIdx.x / kTpr, part = threadIdx.x % kTpr;
        const int ng = ncp / 4;
        float4 m4[kMaxG], z4[kMaxG];
#pragma unroll
        for (int i = 0; i < kMaxG; ++i) {
          const int gi = part + kTpr * i;
          const bool in = r < R && gi < ng;
          m4[i] = in ? __ldcg(reinterpret_cast<const float4*>(pm + static_cast<size_t>(r) * ncp) + gi)
                     : make_float4(kNegBig, kNegBig, kNegBig, kNegBig);
          z4[i] = in ? __ldcg(reinterpret_cast<const float4*>(pz + static_cast<size_t>(r) * ncp) + gi)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mm = kNegBig;
#pragma unroll
        for (int i = 0; i < kMaxG; ++i) mm = fmaxf(mm, fmaxf(fmaxf(m4[i].x, m4[i].y), fmaxf(m4[i].z, m4[i].w)));
#pragma unroll
        for (int o = 1; o < kTpr; o <<= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
        float zz = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxG; ++i)
          zz += z4[i].x * ex2_approx(m4[i].x - mm) + z4[i].y * ex2_approx(m4[i].y - mm) +
                z4[i].z * ex2_approx(m4[i].z - mm) + z4[i].w * ex2_approx(m4[i].w - mm);
#pragma unroll
        for (int o = 1; o < kTpr; o <<= 1) zz += __shfl_xor_sync(0xffffffffu, zz, o);
        if (part == 0 && r < R) {
          // -c2_r / s2 = hi + mid + lo, each part exact in bf16 (about 24 bits in all)
          const float x = -(mm + lg2_approx(zz)) / s2;
          const __nv_bfloat16 hi = __float2bfloat16_rn(x);
          const float x1 = x - __bfloat162float(hi);
          const __nv_bfloat16 mid = __float2bfloat16_rn(x1);
          const __nv_bfloat16 lo = __float2bfloat16_rn(x1 - __bfloat162float(mid));
          const uint32_t w0 = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
                              (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16);
          const uint32_t w1 = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
          uint4* row = reinterpret_cast<uint4*>(sC + r * 32);
          row[0] = make_uint4(w0, w1, 0u, 0u);
          row[1] = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
      }
      fused_epi_bar();
      if (threadIdx.x == 0) mbar_arrive(&c_bar);   // the MMA warp may add the row constants
      // ---------------- epilogue, pass 2 ----------------
      const bool is_max = (a.reduce == 2);
      const float row_scale = (a.reduce == 1) ? 1.f / static_cast<float>(R) : 1.f;
      const size_t out_base = static_cast<size_t>(a.rq.soff[b]) + static_cast<size_t>(h) * n;
      // window rows [ca, ca + 32) of this thread's key, as accumulator values l - c2_r / s2:
      // the causal tail masked, then exp2(x * s2) summed (or x * s2 maximised)
      auto rows32 = [&](float* v, int ca, int wmin, float& acc_sum, float& acc_max) {
        if (wmin > 0) {
          // causal tail: rows whose window position precedes the key do not see it
          int w = ca % W;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (w < wmin) v[j] = -INFINITY;
            w = (w + 1 == W) ? 0 : w + 1;
          }
        }
        if (is_max) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= s2;
          acc_max = fmaxf(acc_max, tree_max<32>(v));
        } else {
          const uint64_t s2p = pack2(s2, s2);
          uint64_t p2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float x0, x1, x2, x3;
            unpack2(fmul2(pack2(v[j + 0], v[j + 1]), s2p), x0, x1);
            unpack2(fmul2(pack2(v[j + 2], v[j + 3]), s2p), x2, x3);
            p2[(j >> 2) & 3] = fadd2(p2[(j >> 2) & 3], pack2(ex2_approx(x0), ex2_approx(x1)));
            p2[(j >> 2) & 3] = fadd2(p2[(j >> 2) & 3], pack2(ex2_approx(x2), ex2_approx(x3)));
          }
          float q0, q1;
          unpack2(fadd2(fadd2(p2[0], p2[1]), fadd2(p2[2], p2[3])), q0, q1);
          acc_sum += q0 + q1;
        }
      };
      if constexpr (MT == 1) {
        // warp (q4, cg) takes tiles cg, cg + 4, ... and sums every window row of its 32 keys
        // alone: rows [0, R/2) from accumulator half 2cg, then rows [R/2, R) from half
        // 2cg + 1, releasing each half as soon as it is summed.  The four warps of a lane
        // quadrant work on different tiles, so their TMEM loads and exponentials
        // interleave on the SM sub-partition, and no warp waits for another.
        for (int t = cg; t < ntiles && alive; t += 4) {
          const int uc = t >> 2;
          const int key = key_begin + t * NT + q4 * 32 + lane;
          const int wmin = a.causal ? key - (n - W) : -1;
          float acc_sum = 0.f, acc_max = -INFINITY;
          for (int hh = 0; hh < 2; ++hh) {
            const int ai = 2 * cg + hh;
            const bool ok = mbar_wait(&accf2[ai], uc & 1, &s_abort, a.wc);
            if (!__all_sync(0xffffffffu, ok)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t trow = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + 128 * cg + 64 * hh;
            const int Rh = R / 2;   // 32 or 64 rows in this half
            float va[32], vb[32];
            tmem_ld32(trow, va);
            tmem_ld_wait();
            if (Rh == 64) {
              tmem_ld32(trow + 32, vb);   // loads while the first 32 rows are summed
              rows32(va, hh * Rh, wmin, acc_sum, acc_max);
              tmem_ld_wait();
              rows32(vb, hh * Rh + 32, wmin, acc_sum, acc_max);
            } else {
              rows32(va, hh * Rh, wmin, acc_sum, acc_max);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce2[ai]);
          }
          if (alive && key < n) a.s_raw[out_base + key] = is_max ? ex2_approx(acc_max) : acc_sum * row_scale;
        }
      } else {
        // R > 128: group g (eight warps) takes tiles g, g+2, ...; the two warps of a lane
        // quadrant split the window rows in halves and add their sums through shared memory
        const int grp = cg >> 1, hf = cg & 1;
        const int Rh = R / 2;   // a multiple of 32
        for (int t = grp; t < ntiles; t += 2) {
          const int acc = t % kAcc2, ua = t / kAcc2;
          const bool ok = mbar_wait(&accf2[acc], ua & 1, &s_abort, a.wc);
          if (!group_all(grp, ok)) break;   // the eight warps of the group leave together
          tc_fence_after();
          const int key = key_begin + t * NT + q4 * 32 + lane;
          const int wmin = a.causal ? key - (n - W) : -1;
          float acc_sum = 0.f, acc_max = -INFINITY;
          const uint32_t trow = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + acc * kAccCols + hf * Rh;
#pragma unroll 1
          for (int c0 = 0; c0 < Rh; c0 += 32) {
            float v[32];
            tmem_ld32(trow + c0, v);
            tmem_ld_wait();
            rows32(v, hf * Rh + c0, wmin, acc_sum, acc_max);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce2[acc]);
          if (hf == 1) s_part[grp][q4 * 32 + lane] = is_max ? acc_max : acc_sum;
          group_bar(grp);
          if (hf == 0 && key < n) {
            const float o = s_part[grp][q4 * 32 + lane];
            a.s_raw[out_base + key] = is_max ? ex2_approx(fmaxf(acc_max, o)) : (acc_sum + o) * row_scale;
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kFMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <int MT, int NT, int STAGES>
cudaError_t launch_rowstats_t(const WinScoreArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t st) {
  const size_t smem = 1024 + 2 * MT * 128 * 128 + STAGES * NT * 256;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(win_rowstats_kernel<MT, NT, STAGES>), smem);
  if (e != cudaSuccess) return e;
  win_rowstats_kernel<MT, NT, STAGES><<<a.ck.total, kThreads, smem, st>>>(tq, tk, a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_win_rowstats(const WinScoreArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, int mt,
                                cudaStream_t st) {
  if (a.ck.total <= 0) return cudaSuccess;
  switch (mt) {
    case 1: return launch_rowstats_t<1, 128, 4>(a, tq, tk, st);
    case 2: return launch_rowstats_t<2, 128, 4>(a, tq, tk, st);
    default: return launch_rowstats_t<4, 64, 4>(a, tq, tk, st);
  }
}

// One cooperative launch for both passes when every chunk's CTA fits on the device at
// once (R <= 256, one CTA per SM); returns cudaErrorNotSupported otherwise.
cudaError_t launch_win_fused(const WinScoreArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                             unsigned int* grid_count, cudaStream_t st) {
  if (a.ck.total <= 0) return cudaSuccess;
  if (a.R > 256 || a.R_pad != a.R || a.R % 64 != 0) return cudaErrorNotSupported;   // 32-row halves
  const int mt = a.R <= 128 ? 1 : 2;
  const void* fn = mt == 1 ? reinterpret_cast<const void*>(win_fused_kernel<1>)
                           : reinterpret_cast<const void*>(win_fused_kernel<2>);
  const size_t smem = 1024 + 2 * static_cast<size_t>(mt) * 128 * 128 + (mt == 1 ? 5 : 4) * 128 * 256 +
                      128 * 32 + static_cast<size_t>(mt) * 128 * 32;   // ones and row constants
  cudaError_t e = ensure_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kFThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1 || a.ck.total > per_sm * sms) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ck.total, 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = mt == 1 ? cudaLaunchKernelEx(&cfg, win_fused_kernel<1>, tq, tk, a, grid_count)
              : cudaLaunchKernelEx(&cfg, win_fused_kernel<2>, tq, tk, a, grid_count);
  if (e == cudaSuccess) note_launch();
  return e;
}

cudaError_t launch_win_keysum(const WinScoreArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t st) {
  if (a.ck.total <= 0) return cudaSuccess;
  const int RP = a.R_pad;
  // accumulators: four (R <= 128) or two (R <= 256), one column group of warps per parity
  const int nacc = RP <= 128 ? 4 : (RP <= 256 ? 2 : 1);
  const uint32_t cols = pow2_cols(static_cast<uint32_t>(nacc * RP));
  const size_t fixed = 1024 + 2 * static_cast<size_t>(RP) * 128 + static_cast<size_t>(RP) * 4;
  const size_t budget = 232448 - 4096;  // opt-in limit minus static shared memory
  int stages = static_cast<int>((budget - fixed) / kKTileBytes);
  stages = stages > 4 ? 4 : stages;
  if (stages < 2) return cudaErrorInvalidValue;
  const size_t smem = fixed + static_cast<size_t>(stages) * kKTileBytes;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(win_keysum_kernel), smem);
  if (e != cudaSuccess) return e;
  win_keysum_kernel<<<a.ck.total, kThreads, smem, st>>>(tq, tk, a, stages, nacc, cols);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
