// Output perturbation of a kept set for the observation-window queries
// ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", Definition 3.1, §3.3 Theorems
//  3.2 and 3.3, App. C.4 Theorem C.1, App. C.5 Table 9).
//
// For a window row r of query head (h, g) with softmax weights A_i over the keys it sees,
// kept set S (of KV head h), kept mass a = sum_{i in S} A_i and projected values
// v'_i = W_O^(h,g) v_i:
//   actual = || W_O^(h,g) sum_i c_i v_i ||_1,  c_i = A_i (1 - [i in S] / a)   (= o - ô)
//   bound  = C - (2 - 1/a) P,  C = sum_i A_i ||v'_i||_1,  P = sum_{i in S} A_i ||v'_i||_1
//   relaxed bound = 2 (1 - a) max_i ||v'_i||_1
//
//   perturb_mask_kernel:   kept positions -> a byte mask.
//   (||v'_i||_1 per query head: the value-norm GEMM, once per group member.)
//   perturb_stats_kernel:  per key chunk, logits Q K^T on tcgen05; each epilogue thread owns
//                          a window row and keeps online max / sums scaled by exp2(l - m):
//                          Z (all keys), Z_S (kept), Z_N (evicted), the evicted and kept
//                          ||v'||_1-weighted sums, and the largest ||v'||_1 it sees.  The
//                          evicted mass is summed on its own (1 - a = Z_N / Z), so nothing
//                          below subtracts two nearly equal masses when a is close to 1.
//   perturb_stats_merge:   chunk partials -> per-row statistics.
//   perturb_accum_kernel:  per key chunk, logits again, c_ri in bf16 high + low parts staged
//                          as the A operand, then E += C V on tcgen05 with V as an MN-major
//                          B operand (the cache tile as TMA writes it).
//   perturb_e_merge:       chunk partials of E, summed in order.
//   perturb_project_kernel / perturb_out_kernel: ||W_O^(h,g) e_r||_1 on CUDA cores (fp32),
//                          then the three outputs.
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr int kPtEpi = 4;                // epilogue warps (thread = window row)
constexpr int kPtProducer = 4;
constexpr int kPtMma = 5;
constexpr int kPtThreads = 192;
constexpr int kPtTile = 128 * 256;       // 128 rows (tokens or window rows) x 128 bf16
constexpr int kPtKStages = 4;            // stats: K tiles in flight
constexpr int kPtKVStages = 2;           // accum: (K, V) tile pairs in flight
constexpr int kPtMaxG = 16;              // group members held in shared memory per tile
constexpr int kPtStat = 7;               // m (log2 units), Z, Z_S, Z_N, C_N, P_S, max ||v'||_1

__device__ __forceinline__ void pt_epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void chunk_of(const ChunkTable& ck, const ReqTable& rq, int cid, int& b, int& h, int& k0,
                                         int& k1) {
  b = 0;
  while (b + 1 < rq.B && ck.base[b + 1] <= cid) ++b;
  const int rem = cid - ck.base[b];
  h = rem / ck.per_head[b];
  const int c = rem - h * ck.per_head[b];
  k0 = c * ck.chunk_len;
  k1 = min(rq.n[b], k0 + ck.chunk_len);
}

// ------------------------------------------------------------------------------------
// kept positions -> byte mask (the mask is zeroed first on the stream)
// ------------------------------------------------------------------------------------
__global__ void perturb_mask_kernel(ReqTable rq, const int32_t* __restrict__ idx, const int32_t* __restrict__ counts,
                                    const int64_t* __restrict__ offsets, uint8_t* __restrict__ keep, int* status) {
  const int seg = blockIdx.y;
  const int b = seg / rq.H, h = seg - b * rq.H;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= __ldg(counts + seg)) return;
  const int n = rq.n[b];
  const int pos = __ldg(idx + __ldg(offsets + seg) + j);
  if (pos < 0 || pos >= n) {
    if (status) atomicOr(status, DEV_BAD_INDEX);
    return;
  }
  keep[rq.soff[b] + static_cast<long long>(h) * n + pos] = 1;
}

}  // namespace

cudaError_t launch_perturb_mask(const ReqTable& rq, const int32_t* idx, const int32_t* counts, const int64_t* offsets,
                                int max_count, uint8_t* keep, int* status, cudaStream_t st) {
  if (max_count <= 0) return cudaSuccess;
  perturb_mask_kernel<<<dim3((max_count + 255) / 256, rq.B * rq.H), 256, 0, st>>>(rq, idx, counts, offsets, keep,
                                                                                  status);
  note_launch();
  return cudaGetLastError();
}

namespace {

// Keys of the 128-key tile starting at tok0 that a window row at position pos sees.
__device__ __forceinline__ int causal_limit(int causal, int pos, int tok0) {
  return causal ? pos - tok0 + 1 : 128;
}

// ------------------------------------------------------------------------------------
// pass 1: per-row statistics of one key chunk
// ------------------------------------------------------------------------------------
// Shared layout: Q [2 K halves][128 rows][128 B], K ring [stages][2][128 keys][128 B].
__global__ void __launch_bounds__(kPtThreads, 1)
    perturb_stats_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const PerturbArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kPtTile;
  __shared__ __align__(8) uint64_t qfull, kfull[kPtKStages], kempty[kPtKStages], accf[2], acce[2], done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ uint8_t s_keep[2][128];
  __shared__ float s_nu[2][kPtMaxG][128];

  const int warp = warp_id(), lane = lane_id();
  int* status = a.wc.status;
  int b, h, k0, k1;
  chunk_of(a.ck, a.rq, blockIdx.x, b, h, k0, k1);
  const int n = a.rq.n[b];
  const int ntiles = (k1 - k0 + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(&qfull, 1);
    for (int s = 0; s < kPtKStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&accf[s], 1);
      mbar_init(&acce[s], kPtEpi);
    }
    mbar_init(&done_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kPtMma) {
    tmem_alloc(&s_tmem, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;

  if (warp == kPtProducer) {
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      const int qrow = (b * a.rq.H + h) * a.R;
      mbar_arrive_expect_tx(&qfull, kPtTile);
      tma_load_2d(sQ, &tq, &qfull, 0, qrow);
      tma_load_2d(sQ + 128 * 128, &tq, &qfull, 64, qrow);
      int t = 0;
      for (; t < ntiles; ++t) {
        const int s = t % kPtKStages;
        if (!mbar_wait(&kempty[s], ((t / kPtKStages) & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&kfull[s], kPtTile);
        load_kv_tile(&tk, a.src, b, h, n, k0 + t * 128, 128, sK + s * kPtTile, &kfull[s], status);
      }
      for (int tt = max(0, t - kPtKStages); tt < t; ++tt) mbar_drain(&kfull[tt % kPtKStages], (tt / kPtKStages) & 1, status);
      mbar_drain(&qfull, 0, status);
      ring_tail(kempty, kPtKStages, t, &s_abort, a.wc);
    }
  } else if (warp == kPtMma) {
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      bool ok = mbar_wait(&qfull, 0, &s_abort, a.wc);
      const uint64_t qdesc = sdesc_kmajor_sw128(smem_u32(sQ));
      for (int t = 0; ok && t < ntiles; ++t) {
        const int s = t % kPtKStages, acc = t & 1;
        if (!mbar_wait(&kfull[s], (t / kPtKStages) & 1, &s_abort, a.wc) ||
            !mbar_wait(&acce[acc], ((t >> 1) & 1) ^ 1, &s_abort, a.wc))
          break;
        tc_fence_after();
        const uint64_t kdesc = sdesc_kmajor_sw128(smem_u32(sK + s * kPtTile));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = ((k >> 2) * (128 * 128) + (k & 3) * 32) >> 4;
          umma_bf16(tbase + acc * 128, qdesc + off, kdesc + off, idesc, k ? 1u : 0u);
        }
        umma_commit(&accf[acc]);
        umma_commit(&kempty[s]);
      }
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, status);
    }
  } else {
    // epilogue: thread r owns window row r (TMEM lane r)
    const int r = threadIdx.x;
    const int g = min(r / max(a.W, 1), a.G - 1);
    const int pos = n - a.W + (r % max(a.W, 1));   // the row's own position
    const bool row_ok = r < a.R;
    float m = -INFINITY, Z = 0.f, ZS = 0.f, ZN = 0.f, CN = 0.f, PS = 0.f, M = 0.f;
    bool ok = true;
    const long long sbase = a.rq.soff[b] + static_cast<long long>(h) * n;
    for (int t = 0; t < ntiles; ++t) {
      const int tok0 = k0 + t * 128;
      const int buf = t & 1;
      // side data of the tile: thread r loads key tok0 + r of every group member
      {
        const int i = tok0 + r;
        const bool in = i < k1;
        s_keep[buf][r] = in ? a.keep[sbase + i] : 0;
        for (int gg = 0; gg < a.G && gg < kPtMaxG; ++gg)
          s_nu[buf][gg][r] = in ? __ldg(a.nu + static_cast<long long>(gg) * a.n_scores + sbase + i) : 0.f;
      }
      pt_epi_bar();
      const int acc = t & 1;
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&accf[acc], (t >> 1) & 1, &s_abort, a.wc));
      float y[128];
      if (ok) {
        tc_fence_after();
        const uint32_t taddr = tbase + (static_cast<uint32_t>(warp * 32) << 16) + acc * 128;
        tmem_ld32(taddr, y);
        tmem_ld32(taddr + 32, y + 32);
        tmem_ld32(taddr + 64, y + 64);
        tmem_ld32(taddr + 96, y + 96);
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[acc]);
      if (ok && row_ok) {
        const int lim = min(k1 - tok0, causal_limit(a.causal, pos, tok0));
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 128; ++j) {
          y[j] *= a.s2;
          if (j < lim) mt = fmaxf(mt, y[j]);
        }
        if (mt > -INFINITY) {
          const float mn = fmaxf(m, mt);
          const float sc = exp2f(m - mn);   // 0 while m is -inf
          Z *= sc;
          ZS *= sc;
          ZN *= sc;
          CN *= sc;
          PS *= sc;
          m = mn;
          const float* nug = s_nu[buf][min(g, kPtMaxG - 1)];
#pragma unroll
          for (int j = 0; j < 128; ++j) {
            if (j < lim) {
              const float e = exp2f(y[j] - m);
              const float nuj = nug[j];
              const bool kept = s_keep[buf][j] != 0;
              Z += e;
              ZS += kept ? e : 0.f;
              ZN += kept ? 0.f : e;
              CN += kept ? 0.f : e * nuj;
              PS += kept ? e * nuj : 0.f;
              M = fmaxf(M, nuj);
            }
          }
        }
      }
    }
    if (row_ok) {
      float* dst = a.stat_part + (static_cast<size_t>(blockIdx.x) * 128 + r) * kPtStat;
      dst[0] = m;
      dst[1] = Z;
      dst[2] = ZS;
      dst[3] = ZN;
      dst[4] = CN;
      dst[5] = PS;
      dst[6] = M;
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kPtMma) {
    tc_fence_after();
    tmem_dealloc(tbase, 256);
  }
}

// Chunk partials of one (request, head) merged per row, chunks in order.
__global__ void perturb_stats_merge(ChunkTable ck, ReqTable rq, int R, const float* __restrict__ part,
                                    float* __restrict__ stat) {
  const int seg = blockIdx.x, r = threadIdx.x;
  if (r >= R) return;
  const int b = seg / rq.H, h = seg - b * rq.H;
  const int c0 = ck.base[b] + h * ck.per_head[b];
  float m = -INFINITY;
  for (int c = 0; c < ck.per_head[b]; ++c) m = fmaxf(m, part[(static_cast<size_t>(c0 + c) * 128 + r) * kPtStat]);
  float acc[5] = {0.f, 0.f, 0.f, 0.f, 0.f}, M = 0.f;
  for (int c = 0; c < ck.per_head[b]; ++c) {
    const float* q = part + (static_cast<size_t>(c0 + c) * 128 + r) * kPtStat;
    const float sc = q[0] > -INFINITY ? exp2f(q[0] - m) : 0.f;
#pragma unroll
    for (int x = 0; x < 5; ++x) acc[x] += q[1 + x] * sc;
    M = fmaxf(M, q[6]);
  }
  float* d = stat + (static_cast<size_t>(seg) * 128 + r) * kPtStat;
  d[0] = m;
#pragma unroll
  for (int x = 0; x < 5; ++x) d[1 + x] = acc[x];
  d[6] = M;
}

// ------------------------------------------------------------------------------------
// pass 2: E = sum_i c_ri v_i over one key chunk
// ------------------------------------------------------------------------------------
// Shared layout: Q [2][128 rows][128 B]; (K, V) ring [stages][K tile, V tile]; C high and
// low parts [2 K halves][128 rows][128 B] each (K-major A operand, keys as K).
constexpr size_t kPtAccumSmem = 1024 + kPtTile + 2 * kPtKVStages * kPtTile + 2 * kPtTile;
constexpr size_t kPtStatsSmem = 1024 + kPtTile + kPtKStages * kPtTile;

// MN-major operand descriptor, 128-byte swizzle: the tile is stored [K rows][64 MN elements
// = 128 B], 8-row atoms 1024 B apart along K (stride byte offset), and the next 64 MN
// elements 16 KB further (leading byte offset: the second half of a 128-wide tile).
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16384u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

__global__ void __launch_bounds__(kPtThreads, 1)
    perturb_accum_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, const PerturbArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kPtTile;                          // stage s: K at 2s, V at 2s + 1
  uint8_t* sC = smem + kPtTile + 2 * kPtKVStages * kPtTile;   // high part, then low part
  __shared__ __align__(8) uint64_t qfull, kvfull[kPtKVStages], kvempty[kPtKVStages], lfull[2], lempty[2];
  __shared__ __align__(8) uint64_t cfull, cempty, efull;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ uint8_t s_keep[2][128];

  const int warp = warp_id(), lane = lane_id();
  int* status = a.wc.status;
  int b, h, k0, k1;
  chunk_of(a.ck, a.rq, blockIdx.x, b, h, k0, k1);
  const int n = a.rq.n[b];
  const int ntiles = (k1 - k0 + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(&qfull, 1);
    for (int s = 0; s < kPtKVStages; ++s) {
      mbar_init(&kvfull[s], 1);
      mbar_init(&kvempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&lfull[s], 1);
      mbar_init(&lempty[s], kPtEpi);
    }
    mbar_init(&cfull, kPtEpi);
    mbar_init(&cempty, 1);
    mbar_init(&efull, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kPtMma) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;            // logits: columns [0, 256); E: [256, 384)
  const uint32_t tE = tbase + 256;

  if (warp == kPtProducer) {
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      const int qrow = (b * a.rq.H + h) * a.R;
      mbar_arrive_expect_tx(&qfull, kPtTile);
      tma_load_2d(sQ, &tq, &qfull, 0, qrow);
      tma_load_2d(sQ + 128 * 128, &tq, &qfull, 64, qrow);
      int t = 0;
      for (; t < ntiles; ++t) {
        const int s = t % kPtKVStages;
        if (!mbar_wait(&kvempty[s], ((t / kPtKVStages) & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&kvfull[s], 2 * kPtTile);
        uint8_t* dk = sKV + (2 * s) * kPtTile;
        load_kv_tile(&tk, a.src, b, h, n, k0 + t * 128, 128, dk, &kvfull[s], status);
        load_kv_tile(&tv, a.src, b, h, n, k0 + t * 128, 128, dk + kPtTile, &kvfull[s], status);
      }
      for (int tt = max(0, t - kPtKVStages); tt < t; ++tt)
        mbar_drain(&kvfull[tt % kPtKVStages], (tt / kPtKVStages) & 1, status);
      mbar_drain(&qfull, 0, status);
      ring_tail(kvempty, kPtKVStages, t, &s_abort, a.wc);
      ring_tail(&cempty, 1, t, &s_abort, a.wc);   // the last tile's C release
    }
  } else if (warp == kPtMma) {
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idesc1 = idesc_bf16_f32(128, 128);
      constexpr uint32_t idesc2 = idesc_bf16_f32(128, 128) | (1u << 16);   // B (V) MN-major
      bool ok = mbar_wait(&qfull, 0, &s_abort, a.wc);
      const uint64_t qdesc = sdesc_kmajor_sw128(smem_u32(sQ));
      const uint64_t chi = sdesc_kmajor_sw128(smem_u32(sC));
      const uint64_t clo = sdesc_kmajor_sw128(smem_u32(sC + kPtTile));
      // E += C(t) V(t): the C tile of t is ready after the epilogue has read logits t
      auto second = [&](int t) -> bool {
        const int s = t % kPtKVStages;
        if (!mbar_wait(&cfull, t & 1, &s_abort, a.wc)) return false;
        tc_fence_after();
        const uint32_t vbase = smem_u32(sKV + (2 * s + 1) * kPtTile);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t aoff = ((k >> 2) * (128 * 128) + (k & 3) * 32) >> 4;
            const uint64_t vdesc = sdesc_mnmajor_sw128(vbase + k * 2048);   // 16 keys per step
            umma_bf16(tE, (part ? clo : chi) + aoff, vdesc, idesc2, (t | part | k) ? 1u : 0u);
          }
        }
        umma_commit(&cempty);
        umma_commit(&kvempty[s]);
        return true;
      };
      int t = 0;
      for (; ok && t < ntiles; ++t) {
        const int s = t % kPtKVStages, acc = t & 1;
        if (!mbar_wait(&kvfull[s], (t / kPtKVStages) & 1, &s_abort, a.wc) ||
            !mbar_wait(&lempty[acc], ((t >> 1) & 1) ^ 1, &s_abort, a.wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kdesc = sdesc_kmajor_sw128(smem_u32(sKV + (2 * s) * kPtTile));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = ((k >> 2) * (128 * 128) + (k & 3) * 32) >> 4;
          umma_bf16(tbase + acc * 128, qdesc + off, kdesc + off, idesc1, k ? 1u : 0u);
        }
        umma_commit(&lfull[acc]);
        if (t > 0 && !second(t - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && ntiles > 0) ok = second(ntiles - 1);
      umma_commit(&efull);
      mbar_drain(&efull, 0, status);
    }
  } else {
    // epilogue: thread r owns window row r (TMEM lane r)
    const int r = threadIdx.x;
    const int pos = n - a.W + (r % max(a.W, 1));
    const bool row_ok = r < a.R;
    const long long sbase = a.rq.soff[b] + static_cast<long long>(h) * n;
    // c_i = A_i (1 - [i kept] / a): 1/Z for an evicted key, -Z_N / (Z Z_S) for a kept one
    float m = 0.f, c_evicted = 0.f, c_kept = 0.f;
    if (row_ok) {
      const float* st = a.stat + (static_cast<size_t>(b * a.rq.H + h) * 128 + r) * kPtStat;
      m = st[0];
      c_evicted = st[1] > 0.f ? 1.f / st[1] : 0.f;
      c_kept = st[2] > 0.f ? -(st[3] / st[2]) * c_evicted : 0.f;
    }
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int tok0 = k0 + t * 128;
      const int buf = t & 1;
      {
        const int i = tok0 + r;
        s_keep[buf][r] = i < k1 ? a.keep[sbase + i] : 0;
      }
      pt_epi_bar();
      const int acc = t & 1;
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&lfull[acc], (t >> 1) & 1, &s_abort, a.wc));
      float y[128];
      if (ok) {
        tc_fence_after();
        const uint32_t taddr = tbase + (static_cast<uint32_t>(warp * 32) << 16) + acc * 128;
        tmem_ld32(taddr, y);
        tmem_ld32(taddr + 32, y + 32);
        tmem_ld32(taddr + 64, y + 64);
        tmem_ld32(taddr + 96, y + 96);
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&lempty[acc]);
      // the C tile of t - 1 has been read by the tensor cores
      if (t > 0) ok = __all_sync(0xffffffffu, ok && mbar_wait(&cempty, (t - 1) & 1, &s_abort, a.wc));
      if (ok) {
        const int lim = row_ok ? min(k1 - tok0, causal_limit(a.causal, pos, tok0)) : 0;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            float c[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int j = q * 8 + e2 * 2 + u;
              c[u] = j < lim ? exp2f(y[j] * a.s2 - m) * (s_keep[buf][j] ? c_kept : c_evicted) : 0.f;
            }
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(c[0], c[1]);
            const float2 hf = __bfloat1622float2(h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(c[0] - hf.x, c[1] - hf.y);
            hi[e2] = *reinterpret_cast<const uint32_t*>(&h2);
            lo[e2] = *reinterpret_cast<const uint32_t*>(&l2);
          }
          const uint32_t off = (q >> 3) * (128 * 128) + r * 128 + (((q & 7) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(sC + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(sC + kPtTile + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&cfull);
    }
    // E rows of this chunk
    ok = __all_sync(0xffffffffu, ok && ntiles > 0 && mbar_wait(&efull, 0, &s_abort, a.wc));
    tc_fence_after();
    if (ok) {
      float* dst = a.e_part + (static_cast<size_t>(blockIdx.x) * 128 + r) * 128;
      for (int c0 = 0; c0 < 128; c0 += 32) {
        float v[32];
        tmem_ld32(tE + (static_cast<uint32_t>(warp * 32) << 16) + c0, v);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kPtMma) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// E of one (request, head): chunk partials summed in order.
__global__ void perturb_e_merge(ChunkTable ck, ReqTable rq, int R, const float* __restrict__ part,
                                float* __restrict__ e) {
  const int seg = blockIdx.x;
  const int b = seg / rq.H, h = seg - b * rq.H;
  const int c0 = ck.base[b] + h * ck.per_head[b];
  for (int x = threadIdx.x; x < R * 128; x += blockDim.x) {
    float acc = 0.f;
    for (int c = 0; c < ck.per_head[b]; ++c) acc += part[static_cast<size_t>(c0 + c) * 128 * 128 + x];
    e[static_cast<size_t>(seg) * 128 * 128 + x] = acc;
  }
}

// ||W_O^(h,g) e_r||_1 over 256 output features per block: thread j holds W_O row j's slice
// of query head (h, g) in fp32 and forms its dot product with every window row of the head;
// the block sums |.| per row.
__global__ void __launch_bounds__(256) perturb_project_kernel(const PerturbArgs a, const uint16_t* __restrict__ w_o) {
  extern __shared__ float s_e[];                    // [W][128]
  __shared__ float s_red[8][128];
  const int bhg = blockIdx.x, slice = blockIdx.y;
  const int G = a.G, W = a.W, H = a.rq.H;
  const int bh = bhg / G, g = bhg - bh * G, h = bh % H;
  const float* e = a.e + (static_cast<size_t>(bh) * 128 + g * W) * 128;
  for (int x = threadIdx.x; x < W * 128; x += 256) s_e[x] = e[x];
  __syncthreads();
  const int j = slice * 256 + threadIdx.x;
  float wr[128];
  const bool jin = j < a.D;
  if (jin) {
    const uint16_t* src = w_o + static_cast<size_t>(j) * H * G * kHeadDim + static_cast<size_t>(h * G + g) * kHeadDim;
#pragma unroll
    for (int c8 = 0; c8 < 16; ++c8) {
      const uint4 p = __ldg(reinterpret_cast<const uint4*>(src) + c8);
      const uint32_t w4[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        wr[c8 * 8 + 2 * u] = __uint_as_float(w4[u] << 16);
        wr[c8 * 8 + 2 * u + 1] = __uint_as_float(w4[u] & 0xFFFF0000u);
      }
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int w = 0; w < W; ++w) {
    float y0 = 0.f, y1 = 0.f, y2 = 0.f, y3 = 0.f;
    if (jin) {
#pragma unroll
      for (int c = 0; c < 128; c += 4) {
        y0 = fmaf(wr[c], s_e[w * 128 + c], y0);
        y1 = fmaf(wr[c + 1], s_e[w * 128 + c + 1], y1);
        y2 = fmaf(wr[c + 2], s_e[w * 128 + c + 2], y2);
        y3 = fmaf(wr[c + 3], s_e[w * 128 + c + 3], y3);
      }
    }
    float v = fabsf((y0 + y1) + (y2 + y3));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) s_red[warp][w & 127] = v;
    if ((w & 127) == 127 || w == W - 1) {
      __syncthreads();
      const int w0 = w & ~127;
      for (int x = threadIdx.x; x <= (w - w0); x += 256) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc += s_red[k][x];
        a.y_part[(static_cast<size_t>(bhg) * gridDim.y + slice) * W + w0 + x] = acc;
      }
      __syncthreads();
    }
  }
}

// The three outputs per window row: actual, bound, relaxed bound.
__global__ void perturb_out_kernel(const PerturbArgs a, int slices) {
  const int bhg = blockIdx.x, w = threadIdx.x;
  if (w >= a.W) return;
  const int G = a.G, W = a.W, H = a.rq.H;
  const int bh = bhg / G, g = bhg - bh * G;
  const int b = bh / H, h = bh - b * H;
  float actual = 0.f;
  for (int s = 0; s < slices; ++s) actual += a.y_part[(static_cast<size_t>(bhg) * slices + s) * W + w];
  const float* st = a.stat + (static_cast<size_t>(bh) * 128 + g * W + w) * kPtStat;
  // with a = Z_S / Z and 1 - a = Z_N / Z:  C - (2 - 1/a) P = (C_N + P_S Z_N / Z_S) / Z
  // (C_N when nothing is kept), and 2 (1 - a) max = 2 (Z_N / Z) max
  const float Z = st[1], ZS = st[2], ZN = st[3], CN = st[4], PS = st[5];
  const float iz = Z > 0.f ? 1.f / Z : 0.f;
  const float bound = (CN + (ZS > 0.f ? PS * (ZN / ZS) : 0.f)) * iz;
  const float relaxed = 2.f * (ZN * iz) * st[6];
  float* o = a.out + static_cast<size_t>(b * H + h) * 3 * G * W + g * W + w;
  o[0] = actual;
  o[static_cast<size_t>(G) * W] = bound;
  o[2 * static_cast<size_t>(G) * W] = relaxed;
}

}  // namespace

cudaError_t launch_perturb_stats(const PerturbArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t st) {
  if (a.ck.total <= 0) return cudaSuccess;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(perturb_stats_kernel), kPtStatsSmem);
  if (e != cudaSuccess) return e;
  perturb_stats_kernel<<<a.ck.total, kPtThreads, kPtStatsSmem, st>>>(tq, tk, a);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  perturb_stats_merge<<<a.rq.B * a.rq.H, 128, 0, st>>>(a.ck, a.rq, a.R, a.stat_part, a.stat);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_perturb_accum(const PerturbArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, cudaStream_t st) {
  if (a.ck.total <= 0) return cudaSuccess;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(perturb_accum_kernel), kPtAccumSmem);
  if (e != cudaSuccess) return e;
  perturb_accum_kernel<<<a.ck.total, kPtThreads, kPtAccumSmem, st>>>(tq, tk, tv, a);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  perturb_e_merge<<<a.rq.B * a.rq.H, 256, 0, st>>>(a.ck, a.rq, a.R, a.e_part, a.e);
  note_launch();
  return cudaGetLastError();
}

int perturb_slices(int D) { return (D + 255) / 256; }

cudaError_t launch_perturb_finish(const PerturbArgs& a, const uint16_t* w_o, cudaStream_t st) {
  const int slices = perturb_slices(a.D);
  const size_t smem = static_cast<size_t>(a.W) * 128 * sizeof(float);
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(perturb_project_kernel), smem);
  if (e != cudaSuccess) return e;
  perturb_project_kernel<<<dim3(a.rq.B * a.rq.H * a.G, slices), 256, smem, st>>>(a, w_o);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  perturb_out_kernel<<<a.rq.B * a.rq.H * a.G, 128, 0, st>>>(a, slices);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
