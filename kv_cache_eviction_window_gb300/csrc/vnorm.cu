// Value norm nu_i = || W_h v_i ||_1 on tcgen05 tensor cores
// ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", §3.4 Algorithm 1: the L1 norm of
//  each row of V W^O; §3.3 Theorem 3.3; App. D.4: a fused pass so the n x D projected
//  values are never stored).
//
// W_h is the D x d output-projection weight seen by KV head h: the sum of the G query
// heads' W_O column slices (one D-vector per token and KV head), or, in the per-head
// reading, the G slices stacked (G*D rows, giving sum_g ||W_O^(h,g) v||_1).
//
//   wbar_kernel: W_h rows in bf16, [H][Dw][d] (sum taken in fp32, rounded once).
//   vnorm_kernel: persistent UMMA GEMM.  A = a block of MSUB*128 value rows (resident in
//     shared memory, double-buffered), B = W_h tiles of NT rows streamed through a TMA
//     ring; accumulators in TMEM are drained by 8 epilogue warps that add |.| along the
//     row, so each thread ends with the L1 norm of one token's projected value.
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;

constexpr int kMsub = 2;                  // 128-token subtiles per work unit
constexpr int kTokBlock = kMsub * 128;    // tokens per work unit
constexpr int kNT = 128;                  // W_h rows per B tile
constexpr int kWStages = 3;
constexpr int kVBuf = 2;
constexpr int kAcc = 2;
constexpr uint32_t kAccCols = kMsub * kNT;        // 256
constexpr uint32_t kTmemCols = kAcc * kAccCols;   // 512
constexpr int kVSub = 128 * 256;                  // bytes of one 128-token subtile
constexpr int kVTile = kMsub * kVSub;
constexpr int kWTile = kNT * 256;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void load_v_rows(const CUtensorMap* map, const KvSource& src, int b, int h, int n,
                                            int tok0, uint8_t* dst, uint64_t* bar, int* status) {
  const int half = 128 * 128;
  if (!src.paged) {
    tma_load_4d(dst, map, bar, 0, tok0, h, b);
    tma_load_4d(dst + half, map, bar, 64, tok0, h, b);
  } else {
    const int bs = src.block_size;
    const int nblk_req = (n + bs - 1) / bs;
    for (int j = 0; j < 128 / bs; ++j) {
      const int lb = tok0 / bs + j;
      int pb = -1;
      if (lb < nblk_req && lb < src.max_blocks) pb = __ldg(src.block_table + (size_t)b * src.max_blocks + lb);
      if (pb < 0 || pb >= src.num_blocks) {
        if (lb < nblk_req) atomicOr(status, DEV_BAD_INDEX);
        pb = 0;
      }
      tma_load_4d(dst + j * bs * 128, map, bar, 0, h, 0, pb);
      tma_load_4d(dst + half + j * bs * 128, map, bar, 64, h, 0, pb);
    }
  }
}

__device__ __forceinline__ void unit_coords(const VnormArgs& a, int u, int& b, int& h, int& blk) {
  b = 0;
  while (b + 1 < a.rq.B && a.unit_base[b + 1] <= u) ++b;
  const int rem = u - a.unit_base[b];
  h = rem / a.blocks_per_head[b];
  blk = rem - h * a.blocks_per_head[b];
}

__global__ void __launch_bounds__(kThreads, 1)
    vnorm_kernel(const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tw, const VnormArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sV = smem;                       // [kVBuf][kMsub][2 halves][128][128 B]
  uint8_t* sW = smem + kVBuf * kVTile;      // [kWStages][2 halves][kNT][128 B]

  __shared__ __align__(8) uint64_t wfull[kWStages], wempty[kWStages], vfull[kVBuf], vempty[kVBuf];
  __shared__ __align__(8) uint64_t accf[kAcc], acce[kAcc], done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = warp_id(), lane = lane_id();
  int* status = a.wc.status;
  const int nwt = a.Dw / kNT;   // W tiles per unit

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 1);
    }
    for (int s = 0; s < kVBuf; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int s = 0; s < kAcc; ++s) {
      mbar_init(&accf[s], 1);
      mbar_init(&acce[s], kEpiWarps);
    }
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
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tw);
      int wt = 0;     // W tiles issued so far (global across units)
      int iu = 0;     // units processed by this CTA
      bool ok = true;
      int last_v = -1;
      for (int u = blockIdx.x; ok && u < a.units_total; u += gridDim.x, ++iu) {
        int b, h, blk;
        unit_coords(a, u, b, h, blk);
        const int n = a.rq.n[b];
        const int vb = iu % kVBuf, vu = iu / kVBuf;
        if (!mbar_wait(&vempty[vb], (vu & 1) ^ 1, &s_abort, a.wc)) break;
        mbar_arrive_expect_tx(&vfull[vb], kVTile);
        for (int m = 0; m < kMsub; ++m)
          load_v_rows(&tv, a.src, b, h, n, blk * kTokBlock + m * 128, sV + vb * kVTile + m * kVSub, &vfull[vb],
                      status);
        last_v = iu;
        for (int j = 0; j < nwt; ++j, ++wt) {
          const int s = wt % kWStages, us = wt / kWStages;
          if (!mbar_wait(&wempty[s], (us & 1) ^ 1, &s_abort, a.wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&wfull[s], kWTile);
          tma_load_3d(sW + s * kWTile, &tw, &wfull[s], 0, j * kNT, h);
          tma_load_3d(sW + s * kWTile + kNT * 128, &tw, &wfull[s], 64, j * kNT, h);
        }
      }
      for (int tt = max(0, wt - kWStages); tt < wt; ++tt) mbar_drain(&wfull[tt % kWStages], (tt / kWStages) & 1, status);
      for (int vv = max(0, last_v - kVBuf + 1); vv <= last_v; ++vv)
        mbar_drain(&vfull[vv % kVBuf], (vv / kVBuf) & 1, status);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kNT);
      int wt = 0, t = 0, iu = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.units_total; u += gridDim.x, ++iu) {
        const int vb = iu % kVBuf, vu = iu / kVBuf;
        if (!mbar_wait(&vfull[vb], vu & 1, &s_abort, a.wc)) break;
        const uint32_t vbase = smem_u32(sV + vb * kVTile);
        for (int j = 0; j < nwt; ++j, ++wt, ++t) {
          const int s = wt % kWStages, us = wt / kWStages;
          const int acc = t % kAcc, ua = t / kAcc;
          if (!mbar_wait(&wfull[s], us & 1, &s_abort, a.wc) ||
              !mbar_wait(&acce[acc], (ua & 1) ^ 1, &s_abort, a.wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t wbase = smem_u32(sW + s * kWTile);
#pragma unroll
          for (int m = 0; m < kMsub; ++m) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t koff = (k & 3) * 32;
              const uint64_t da = sdesc_kmajor_sw128(vbase + m * kVSub + (k >> 2) * (128 * 128) + koff);
              const uint64_t db = sdesc_kmajor_sw128(wbase + (k >> 2) * (kNT * 128) + koff);
              umma_bf16(tbase + acc * kAccCols + m * kNT, da, db, idesc, k > 0 ? 1u : 0u);
            }
          }
          umma_commit(&wempty[s]);
          umma_commit(&accf[acc]);
        }
        if (ok) umma_commit(&vempty[vb]);
      }
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, status);
    }
  } else {
    // epilogue: warp e owns TMEM lane quadrant e%4 of subtile e/4
    const int q4 = warp & 3, m = warp >> 2;
    int t = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.units_total; u += gridDim.x) {
      int b, h, blk;
      unit_coords(a, u, b, h, blk);
      const int n = a.rq.n[b];
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      for (int j = 0; j < nwt; ++j, ++t) {
        const int acc = t % kAcc, ua = t / kAcc;
        bool w = mbar_wait(&accf[acc], ua & 1, &s_abort, a.wc);
        w = __all_sync(0xffffffffu, w);
        if (!w) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + acc * kAccCols + m * kNT;
#pragma unroll
        for (int c0 = 0; c0 < kNT; c0 += 64) {
          float v[64];
          tmem_ld32(taddr + c0, v);
          tmem_ld32(taddr + c0 + 32, v + 32);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 64; i += 4) {
            s0 += fabsf(v[i + 0]);
            s1 += fabsf(v[i + 1]);
            s2 += fabsf(v[i + 2]);
            s3 += fabsf(v[i + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[acc]);
      }
      if (!ok) break;
      const int tok = blk * kTokBlock + m * 128 + q4 * 32 + lane;
      if (tok < n) a.nu[a.rq.soff[b] + static_cast<size_t>(h) * n + tok] = (s0 + s1) + (s2 + s3);
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

// W_h[h][j][c]: group sum of W_O[j][(h*G+g)*d + c] (wo_mode 0) or the stacked slices
// W_h[h][g*D + j][c] = W_O[j][(h*G+g)*d + c] (wo_mode 1).  One thread per 8 columns.
__global__ void wbar_kernel(const uint16_t* __restrict__ w_o, uint16_t* __restrict__ wbar, int H, int G, int D,
                            int wo_mode) {
  const long long total = static_cast<long long>(H) * D * 16;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long row_len = static_cast<long long>(H) * G * kHeadDim;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total; t += stride) {
    const int c8 = static_cast<int>(t % 16);
    const long long hj = t / 16;
    const int j = static_cast<int>(hj % D);
    const int h = static_cast<int>(hj / D);
    const uint16_t* src = w_o + j * row_len + static_cast<long long>(h) * G * kHeadDim + c8 * 8;
    if (wo_mode == 0) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int g = 0; g < G; ++g) {
        const uint4 p = __ldg(reinterpret_cast<const uint4*>(src + g * kHeadDim));
        const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] += __uint_as_float(w[i] << 16);
          acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 r = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t*>(&r);
      }
      *reinterpret_cast<uint4*>(wbar + (static_cast<long long>(h) * D + j) * kHeadDim + c8 * 8) =
          make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      for (int g = 0; g < G; ++g) {
        const uint4 p = __ldg(reinterpret_cast<const uint4*>(src + g * kHeadDim));
        *reinterpret_cast<uint4*>(wbar + ((static_cast<long long>(h) * G + g) * D + j) * kHeadDim + c8 * 8) = p;
      }
    }
  }
}

}  // namespace

int vnorm_token_block() { return kTokBlock; }
int vnorm_w_tile_rows() { return kNT; }

cudaError_t launch_wbar(const uint16_t* w_o, uint16_t* wbar, int H, int G, int D, int wo_mode, cudaStream_t st) {
  const long long total = static_cast<long long>(H) * D * 16;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  wbar_kernel<<<static_cast<unsigned>(blocks < 65535 * 8 ? blocks : 65535 * 8), threads, 0, st>>>(w_o, wbar, H, G, D,
                                                                                                  wo_mode);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_vnorm(const VnormArgs& a, const CUtensorMap& tv, const CUtensorMap& tw, cudaStream_t st) {
  if (a.units_total <= 0) return cudaSuccess;
  const size_t smem = 1024 + kVBuf * kVTile + kWStages * kWTile;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(vnorm_kernel), smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.units_total < sms ? a.units_total : sms;
  vnorm_kernel<<<grid, kThreads, smem, st>>>(tv, tw, a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
