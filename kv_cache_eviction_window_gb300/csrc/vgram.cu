// L2 value norm through the d x d Gram matrix of the output projection
// ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", App. C.3: the Euclidean
//  distance as the alternative to L1; same page §3.3 Theorem 3.3 for the projected value).
//
// ||W_h v||_2^2 = v^T (W_h^T W_h) v, so with the d x d Gram matrix Gamma_h = W_h^T W_h the
// per-token cost drops from 2*D*d to 2*d*d flop (D / d = 32x for a 4096-wide model):
//
//   gram_fused_kernel: Gamma_h partials straight from W_O: per 256-row slice, the group
//                      sum of the W_O columns of head h in fp32 (the same values wbar_kernel
//                      rounds), rounded once to bf16 and transposed in shared memory into
//                      a K-major operand, then A = B = that operand on tcgen05 (M = N =
//                      128, K = 64 per batch); W_h^T is never written to memory.
//   gram_finish_kernel: Gamma_h = sum of the partials (fixed order), split into a bf16 high
//                      part and a bf16 remainder so the tensor cores see it to ~2^-16.
//   vgram_kernel:      persistent: per 128-token tile, Y = V (Gamma_hi + Gamma_lo) on tcgen05
//                      (16 UMMAs into one TMEM accumulator), then each epilogue thread
//                      forms nu = sqrt(sum_c Y[c] v[c]) for its token, reading v from the
//                      same shared-memory tile.
#include "internal.cuh"

namespace kvsel {
namespace {


// ------------------------------------------------------------------------------------
// Gamma partials straight from W_O (group sum, transpose and W^T W in one kernel)
// ------------------------------------------------------------------------------------
// Block (slice s, head h): rows [s * 256, s * 256 + 256) of W_O in batches of 64.  Per
// batch the G column slices of head h arrive by TMA (128-byte swizzle); eight worker warps
// sum them in fp32 into a padded tile [64 rows j][129], then write it transposed and
// rounded to bf16 as a K-major operand [128 columns c][64 j]; one thread issues
// D[c][c'] += sum_j A[c][j] A[c'][j] (four K = 16 UMMAs).  W_h^T never reaches memory.
constexpr int kGfRows = 256;                 // W_O rows per CTA
constexpr int kGfBatch = 64;                 // rows per batch (UMMA K per batch)
constexpr int kGfWorkers = 256;
constexpr int kGfThreads = kGfWorkers + 32;
constexpr int kGfBox = kGfBatch * 128;       // one TMA box: 64 rows x 64 columns bf16
constexpr int kGfA = 128 * 128;              // operand: 128 rows c x 64 j bf16 (128 B rows)
constexpr int kGfTileStride = 129;           // fp32 tile row stride (conflict-free transposes)

__device__ __forceinline__ void gf_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__global__ void __launch_bounds__(kGfThreads, 1)
    gram_fused_kernel(const __grid_constant__ CUtensorMap two, float* part, int G, int D, int raw_stages, WaitCtl wc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const int raw_bytes = G * 2 * kGfBox;                  // one batch: G slices x 2 column halves
  uint8_t* sRaw = smem;                                  // [raw_stages][G][2][64 rows][128 B]
  uint8_t* sA = smem + raw_stages * raw_bytes;           // [2][128 c][128 B]
  float* ft = reinterpret_cast<float*>(sA + 2 * kGfA);   // [64][129] fp32
  __shared__ __align__(8) uint64_t rfull[2], rempty[2], afull[2], aempty[2], done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = warp_id(), lane = lane_id();
  const int s = blockIdx.x, h = blockIdx.y;
  const int row0 = s * kGfRows;
  const int nb = min(kGfRows, D - row0) > 0 ? (min(kGfRows, D - row0) + kGfBatch - 1) / kGfBatch : 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], kGfWorkers / 32);
      mbar_init(&afull[i], kGfWorkers / 32);
      mbar_init(&aempty[i], 1);
    }
    mbar_init(&done_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(&s_tmem, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;

  if (warp == 8) {
    if (lane == 0 && nb > 0) {
      tma_prefetch_desc(&two);
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      // the producer runs ahead by raw_stages batches; the MMA of batch t follows the
      // workers' transpose of batch t
      int issued = 0;
      auto load = [&](int t) -> bool {
        const int rs = t % raw_stages;
        if (t >= raw_stages && !mbar_wait(&rempty[rs], ((t / raw_stages) & 1) ^ 1, &s_abort, wc)) return false;
        mbar_arrive_expect_tx(&rfull[rs], raw_bytes);
        uint8_t* dst = sRaw + rs * raw_bytes;
        for (int g = 0; g < G; ++g)
          for (int x = 0; x < 2; ++x)
            tma_load_2d(dst + (g * 2 + x) * kGfBox, &two, &rfull[rs], (h * G + g) * 128 + x * 64, row0 + t * kGfBatch);
        return true;
      };
      bool ok = true;
      for (; ok && issued < min(nb, raw_stages); ++issued) ok = load(issued);
      for (int t = 0; ok && t < nb; ++t) {
        const int as = t & 1;
        if (!mbar_wait(&afull[as], (t >> 1) & 1, &s_abort, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(sA + as * kGfA));
#pragma unroll
        for (int k = 0; k < 4; ++k) umma_bf16(tbase, adesc + ((k * 32) >> 4), adesc + ((k * 32) >> 4), idesc, (t | k) ? 1u : 0u);
        umma_commit(&aempty[as]);
        if (issued < nb) ok = load(issued++);
      }
      // drain copies still in flight
      for (int t = max(0, issued - raw_stages); t < issued; ++t) mbar_drain(&rfull[t % raw_stages], (t / raw_stages) & 1, wc.status);
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, wc.status);
      ring_tail(aempty, 2, nb, &s_abort, wc);
    }
  } else {
    const int tid = threadIdx.x;
    bool ok = true;
    for (int t = 0; t < nb; ++t) {
      const int rs = t % raw_stages, as = t & 1;
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&rfull[rs], (t / raw_stages) & 1, &s_abort, wc));
      const uint8_t* raw = sRaw + rs * raw_bytes;
      if (ok) {
        // step 1: thread (row j = lane + 32 * (warp & 1), 16-byte chunk q) sums the G slices
        for (int it = 0; it < 4; ++it) {
          const int j = lane + 32 * (warp & 1);
          const int q = (warp >> 1) + 4 * it;   // 0..15: column chunk of 8
          float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int g = 0; g < G; ++g) {
            const uint8_t* box = raw + (g * 2 + (q >> 3)) * kGfBox;
            const uint4 p = *reinterpret_cast<const uint4*>(box + j * 128 + (((q & 7) ^ (j & 7)) << 4));
            const uint32_t w4[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[2 * e] += __uint_as_float(w4[e] << 16);
              acc[2 * e + 1] += __uint_as_float(w4[e] & 0xFFFF0000u);
            }
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) ft[j * kGfTileStride + q * 8 + e] = acc[e];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[rs]);   // the raw stage may be refilled
      gf_bar();                                   // the fp32 tile is complete
      // the operand buffer was last read by the UMMAs of batch t - 2
      if (t >= 2) ok = __all_sync(0xffffffffu, ok && mbar_wait(&aempty[as], ((t >> 1) & 1) ^ 1, &s_abort, wc));
      if (ok) {
        // step 2: thread (column c = tid & 127, 8-row chunk jc) writes 8 rounded values of
        // row c of the K-major operand
        for (int it = 0; it < 4; ++it) {
          const int c = tid & 127;
          const int jc = (tid >> 7) + 2 * it;   // 0..7
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(ft[(jc * 8 + 2 * e) * kGfTileStride + c],
                                                            ft[(jc * 8 + 2 * e + 1) * kGfTileStride + c]);
            o[e] = *reinterpret_cast<const uint32_t*>(&v2);
          }
          *reinterpret_cast<uint4*>(sA + as * kGfA + c * 128 + ((jc ^ (c & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[as]);
      gf_bar();                                   // the fp32 tile may be overwritten
    }
    // epilogue: warps 0-3 own the accumulator's lanes
    if (warp < 4) {
      ok = __all_sync(0xffffffffu, ok && nb > 0 && mbar_wait(&done_bar, 0, &s_abort, wc));
      tc_fence_after();
      if (ok) {
        float* dst = part + ((static_cast<size_t>(h) * gridDim.x + s) * 128 + warp * 32 + lane) * 128;
        for (int c0 = 0; c0 < 128; c0 += 32) {
          float v[32];
          tmem_ld32(tbase + (static_cast<uint32_t>(warp * 32) << 16) + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      } else if (nb == 0) {
        float* dst = part + ((static_cast<size_t>(h) * gridDim.x + s) * 128 + warp * 32 + lane) * 128;
        for (int c0 = 0; c0 < 128; ++c0) dst[c0] = 0.f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 128);
  }
}

// Gamma_h = sum_s partial[h][s] (in order), split: hi = bf16(Gamma), lo = bf16(Gamma - hi).
// Output [H][2][128][128] bf16; row n of either matrix is the K-major B operand row n.
__global__ void __launch_bounds__(256) gram_finish_kernel(const float* __restrict__ part, uint16_t* __restrict__ gam,
                                                          int S) {
  const int h = blockIdx.y;
  for (int e = blockIdx.x * 256 + threadIdx.x; e < 128 * 128; e += gridDim.x * 256) {
    // eight partials loaded before they are added (in order), so the loads overlap
    const float* src = part + static_cast<size_t>(h) * S * 128 * 128 + e;
    float g = 0.f;
    int s = 0;
    for (; s + 8 <= S; s += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldg(src + static_cast<size_t>(s + u) * 128 * 128);
#pragma unroll
      for (int u = 0; u < 8; ++u) g += v[u];
    }
    for (; s < S; ++s) g += __ldg(src + static_cast<size_t>(s) * 128 * 128);
    const __nv_bfloat16 hi = __float2bfloat16_rn(g);
    const __nv_bfloat16 lo = __float2bfloat16_rn(g - __bfloat162float(hi));
    gam[(static_cast<size_t>(h) * 2 + 0) * 128 * 128 + e] = *reinterpret_cast<const uint16_t*>(&hi);
    gam[(static_cast<size_t>(h) * 2 + 1) * 128 * 128 + e] = *reinterpret_cast<const uint16_t*>(&lo);
  }
}

// ------------------------------------------------------------------------------------
// nu = sqrt(v^T Gamma v)
// ------------------------------------------------------------------------------------
constexpr int kVgEpiWarps = 4;
constexpr int kVgProducer = 4;
constexpr int kVgMma = 5;
constexpr int kVgThreads = 192;
constexpr int kVgStages = 4;
constexpr int kVgTile = 128 * 256;     // 128 tokens x 128 bf16
constexpr int kVgGamma = 128 * 256;    // one 128 x 128 bf16 matrix
constexpr int kVgAcc = 2;

__device__ __forceinline__ void vg_unit(const VgramArgs& a, int u, int& b, int& h, int& blk) {
  b = 0;
  while (b + 1 < a.rq.B && a.unit_base[b + 1] <= u) ++b;
  const int rem = u - a.unit_base[b];
  h = rem / a.blocks_per_head[b];
  blk = rem - h * a.blocks_per_head[b];
}

__global__ void __launch_bounds__(kVgThreads, 1)
    vgram_kernel(const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg, const VgramArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sG = smem;                   // [hi, lo][2 K halves][128 rows][128 B]
  uint8_t* sV = smem + 2 * kVgGamma;    // [stages][2 K halves][128 tokens][128 B]

  __shared__ __align__(8) uint64_t vfull[kVgStages], vempty[kVgStages], accf[kVgAcc], acce[kVgAcc];
  __shared__ __align__(8) uint64_t gfull, gempty, done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = warp_id(), lane = lane_id();
  int* status = a.wc.status;
  const int lo = static_cast<int>(static_cast<long long>(blockIdx.x) * a.units_total / gridDim.x);
  const int hi = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * a.units_total / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kVgStages; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], kVgEpiWarps);
    }
    for (int s = 0; s < kVgAcc; ++s) {
      mbar_init(&accf[s], 1);
      mbar_init(&acce[s], kVgEpiWarps);
    }
    mbar_init(&gfull, 1);
    mbar_init(&gempty, 1);
    mbar_init(&done_bar, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kVgMma) {
    tmem_alloc(&s_tmem, kVgAcc * 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;

  if (warp == kVgProducer) {
    if (lane == 0 && hi > lo) {
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tg);
      int cur_h = -1, gl = 0, t = 0;
      for (int u = lo; u < hi; ++u, ++t) {
        int b, h, blk;
        vg_unit(a, u, b, h, blk);
        if (h != cur_h) {
          // the previous head's Gamma is released by the UMMA warp after its last tile
          if (gl > 0 && !mbar_wait(&gempty, (gl - 1) & 1, &s_abort, a.wc)) break;
          mbar_arrive_expect_tx(&gfull, 2 * kVgGamma);
          for (int m = 0; m < 2; ++m) {
            tma_load_2d(sG + m * kVgGamma, &tg, &gfull, 0, (h * 2 + m) * 128);
            tma_load_2d(sG + m * kVgGamma + 128 * 128, &tg, &gfull, 64, (h * 2 + m) * 128);
          }
          cur_h = h;
          ++gl;
        }
        const int s = t % kVgStages, us = t / kVgStages;
        if (!mbar_wait(&vempty[s], (us & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&vfull[s], kVgTile);
        load_kv_tile(&tv, a.src, b, h, a.rq.n[b], blk * 128, 128, sV + s * kVgTile, &vfull[s], status);
      }
      // drain copies still in flight
      for (int tt = max(0, t - kVgStages); tt < t; ++tt) mbar_drain(&vfull[tt % kVgStages], (tt / kVgStages) & 1, status);
      if (gl > 0) mbar_drain(&gfull, (gl - 1) & 1, status);
      ring_tail(&gempty, 1, gl, &s_abort, a.wc);   // the last Gamma's release (V stages are released by threads)
    }
  } else if (warp == kVgMma) {
    if (lane == 0 && hi > lo) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint64_t gdesc[2] = {sdesc_kmajor_sw128(smem_u32(sG)), sdesc_kmajor_sw128(smem_u32(sG + kVgGamma))};
      int cur_h = -1, gl = 0, t = 0;
      bool ok = true;
      for (int u = lo; ok && u < hi; ++u, ++t) {
        int b, h, blk;
        vg_unit(a, u, b, h, blk);
        if (h != cur_h) {
          if (!mbar_wait(&gfull, gl & 1, &s_abort, a.wc)) break;
          cur_h = h;
          ++gl;
        }
        const int s = t % kVgStages, us = t / kVgStages;
        const int acc = t % kVgAcc, ua = t / kVgAcc;
        if (!mbar_wait(&vfull[s], us & 1, &s_abort, a.wc) || !mbar_wait(&acce[acc], (ua & 1) ^ 1, &s_abort, a.wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t vdesc = sdesc_kmajor_sw128(smem_u32(sV + s * kVgTile));
#pragma unroll
        for (int m = 0; m < 2; ++m) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = ((k >> 2) * (128 * 128) + (k & 3) * 32) >> 4;
            umma_bf16(tbase + acc * 128, vdesc + off, gdesc[m] + off, idesc, (m | k) ? 1u : 0u);
          }
        }
        umma_commit(&accf[acc]);
        // the head changes after this tile (or the range ends): its Gamma may be replaced
        int nb, nh, nblk;
        if (u + 1 < hi) vg_unit(a, u + 1, nb, nh, nblk);
        if (u + 1 >= hi || nh != h) umma_commit(&gempty);
      }
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, status);
    }
  } else {
    // epilogue: warp q4 owns TMEM lanes / tokens [32 q4, 32 q4 + 32) of each tile
    const int q4 = warp;
    const int r = q4 * 32 + lane;
    int t = 0;
    for (int u = lo; u < hi; ++u, ++t) {
      int b, h, blk;
      vg_unit(a, u, b, h, blk);
      const int s = t % kVgStages;
      const int acc = t % kVgAcc, ua = t / kVgAcc;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&accf[acc], ua & 1, &s_abort, a.wc));
      if (!ok) break;
      tc_fence_after();
      const uint8_t* vrow = sV + s * kVgTile + r * 128;
      float dp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // independent partial sums
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 64) {
        float y[64];
        const uint32_t taddr = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + acc * 128 + c0;
        tmem_ld32(taddr, y);
        tmem_ld32(taddr + 32, y + 32);
        tmem_ld_wait();
        // columns c0 .. c0+63 pair with v elements c0 .. c0+63: K half c0/64, eight 16-byte
        // chunks of row r, 128-byte swizzled (chunk q at q ^ (r % 8))
        const uint8_t* half = vrow + (c0 / 64) * (128 * 128);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w = *reinterpret_cast<const uint4*>(half + ((q ^ (r & 7)) << 4));
          const uint32_t e[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            dp[2 * i] = fmaf(y[q * 8 + 2 * i], __uint_as_float(e[i] << 16), dp[2 * i]);
            dp[2 * i + 1] = fmaf(y[q * 8 + 2 * i + 1], __uint_as_float(e[i] & 0xFFFF0000u), dp[2 * i + 1]);
          }
        }
      }
      const float dot = ((dp[0] + dp[1]) + (dp[2] + dp[3])) + ((dp[4] + dp[5]) + (dp[6] + dp[7]));
      // accumulator and value stage are both read: hand them back
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&acce[acc]);
        mbar_arrive(&vempty[s]);
      }
      const int n = a.rq.n[b];
      const int tok = blk * 128 + r;
      if (tok < n) a.nu[a.rq.soff[b] + static_cast<size_t>(h) * n + tok] = sqrtf(fmaxf(dot, 0.f));
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kVgMma) {
    tc_fence_after();
    tmem_dealloc(tbase, kVgAcc * 128);
  }
}

}  // namespace

// Slices of W_O rows per head in the Gamma partials: one per 256 rows.
int gram_slices(int Dw) { return (Dw + kGfRows - 1) / kGfRows; }

cudaError_t launch_value_gram(const CUtensorMap& two, float* part, uint16_t* gam, int H, int G, int D, WaitCtl wc,
                              cudaStream_t st) {
  const int S = gram_slices(D);
  const int raw_stages = G <= 4 ? 2 : 1;
  const size_t smem = 1024 + static_cast<size_t>(raw_stages) * G * 2 * kGfBox + 2 * kGfA +
                      static_cast<size_t>(kGfBatch) * kGfTileStride * sizeof(float);
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(gram_fused_kernel), smem);
  if (e != cudaSuccess) return e;
  gram_fused_kernel<<<dim3(S, H), kGfThreads, smem, st>>>(two, part, G, D, raw_stages, wc);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gram_finish_kernel<<<dim3(64, H), 256, 0, st>>>(part, gam, S);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_vgram(const VgramArgs& a, const CUtensorMap& tv, const CUtensorMap& tg, cudaStream_t st) {
  if (a.units_total <= 0) return cudaSuccess;
  const size_t smem = 1024 + 2 * kVgGamma + kVgStages * kVgTile;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(vgram_kernel), smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (a.grid_cap > 0 && a.grid_cap < sms) sms = a.grid_cap;
  const int grid = a.units_total < sms ? a.units_total : sms;
  vgram_kernel<<<grid, kVgThreads, smem, st>>>(tv, tg, a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
