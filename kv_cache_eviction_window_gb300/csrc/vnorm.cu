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
//   vnorm_kernel: persistent UMMA GEMM, M = 128 value rows (a subtile), N = 256 W_h rows,
//     K = d = 128.  A work unit is 256 tokens of one (request, head): its two subtiles
//     stay in shared memory while all W_h tiles stream through a two-stage TMA ring, and
//     each round (W tile j, subtile m) accumulates into TMEM accumulator m.  Eight
//     epilogue warps drain the accumulators adding |.| along the row, so each thread ends
//     with half the L1 norm of one token's projected value; the halves meet in shared
//     memory.
//
// With K = 128 every round is only eight UMMAs; the tensor pipe queues just a few, so the
// issuing thread's barrier waits and commits between rounds are hidden only when each
// UMMA is long: hence N = 256 (128 cycles per UMMA) rather than 128.  The shared memory
// this takes leaves room for a single value buffer, which the epilogue threads refill:
// each holds the next unit's row of one token in registers (loaded early with plain
// loads) and writes it, 128-byte swizzled, as soon as the last round reading that subtile
// has completed.
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;

constexpr int kMsub = 2;                  // 128-token subtiles per work unit
constexpr int kTokBlock = kMsub * 128;    // tokens per work unit
constexpr int kNT = 256;                  // W_h rows per B tile (UMMA N)
constexpr int kWStages = 2;
constexpr uint32_t kAccCols = kNT;                // accumulator of one subtile
constexpr uint32_t kTmemCols = kMsub * kAccCols;  // 512
constexpr int kVSub = 128 * 256;                  // bytes of one 128-token subtile
constexpr int kVTile = kMsub * kVSub;
constexpr int kWTile = kNT * 256;
constexpr int kEpiCols = kNT / 2;                 // accumulator columns per epilogue warp

__device__ __forceinline__ void unit_coords(const VnormArgs& a, int u, int& b, int& h, int& blk) {
  b = 0;
  while (b + 1 < a.rq.B && a.unit_base[b + 1] <= u) ++b;
  const int rem = u - a.unit_base[b];
  h = rem / a.blocks_per_head[b];
  blk = rem - h * a.blocks_per_head[b];
}

// Work balance: the items (unit, W tile) of the whole launch, unit-major, are cut into
// gridDim.x equal contiguous ranges.  A CTA's range splits into segments, one per unit
// it touches; a unit shared by two CTAs gets its L1 norm in two parts, added atomically
// into nu (zeroed beforehand; with two terms the sum does not depend on their order).
struct Seg {
  int u, j0, j1;
};
__device__ __forceinline__ void cta_items(int total, int& lo, int& hi) {
  lo = static_cast<int>(static_cast<long long>(blockIdx.x) * total / gridDim.x);
  hi = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * total / gridDim.x);
}
__device__ __forceinline__ int seg_count(int lo, int hi, int nwt) {
  return hi > lo ? (hi - 1) / nwt - lo / nwt + 1 : 0;
}
__device__ __forceinline__ Seg seg_at(int lo, int hi, int nwt, int q) {
  Seg g;
  g.u = lo / nwt + q;
  g.j0 = max(lo - g.u * nwt, 0);
  g.j1 = min(hi - g.u * nwt, nwt);
  return g;
}

// One token's value row (128 bf16) of unit u, subtile m, row r into registers; zeros past
// the request's end or for a block-table entry out of range (flagged).
__device__ __forceinline__ void load_v_row(const VnormArgs& a, int u, int m, int r, uint4 (&row)[16]) {
  int b, h, blk;
  unit_coords(a, u, b, h, blk);
  const int n = a.rq.n[b];
  const int tok = blk * kTokBlock + m * 128 + r;
  const uint4* src = nullptr;
  if (tok < n) {
    if (!a.src.paged) {
      src = reinterpret_cast<const uint4*>(a.v + b * a.stride_req + h * a.stride_head +
                                           static_cast<long long>(tok) * a.stride_tok);
    } else {
      const int bs = a.src.block_size;
      const int pb = __ldg(a.src.block_table + static_cast<size_t>(b) * a.src.max_blocks + tok / bs);
      if (pb >= 0 && pb < a.src.num_blocks)
        src = reinterpret_cast<const uint4*>(a.v + ((static_cast<long long>(pb) * bs + tok % bs) * a.rq.H + h) *
                                                       kHeadDim);
      else if (a.wc.status)
        atomicOr(a.wc.status, DEV_BAD_INDEX);
    }
  }
#pragma unroll
  for (int q = 0; q < 16; ++q) row[q] = src ? __ldcs(src + q) : make_uint4(0, 0, 0, 0);
}

// The row into a K-major, 128-byte-swizzled subtile [2 K halves][128 rows][128 B]: the
// 16-byte chunk c of row r sits at chunk c ^ (r % 8) of the row (the TMA SWIZZLE_128B
// pattern, which the UMMA descriptor expects).
__device__ __forceinline__ void store_v_row(uint8_t* sub, int r, const uint4 (&row)[16]) {
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int kh = q >> 3, c = q & 7;
    *reinterpret_cast<uint4*>(sub + kh * (128 * 128) + r * 128 + ((c ^ (r & 7)) << 4)) = row[q];
  }
}

__device__ __forceinline__ bool epi_vote_any(bool pred) {
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

__global__ void __launch_bounds__(kThreads, 1)
    vnorm_kernel(const __grid_constant__ CUtensorMap tw, const VnormArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint8_t* sV = smem;                // [kMsub][2 K halves][128 rows][128 B]
  uint8_t* sW = smem + kVTile;       // [kWStages][2 K halves][kNT rows][128 B]

  __shared__ __align__(8) uint64_t wfull[kWStages], wempty[kWStages], vfull[kMsub];
  __shared__ __align__(8) uint64_t accf[kMsub], acce[kMsub], done_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_half[kMsub][128];

  const int warp = warp_id(), lane = lane_id();
  int* status = a.wc.status;
  const int nwt = (a.Dw + kNT - 1) / kNT;   // W tiles per unit (rows past Dw read as zeros)
  int lo, hi;
  cta_items(a.units_total * nwt, lo, hi);
  const int nseg = seg_count(lo, hi, nwt);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 1);
    }
    for (int m = 0; m < kMsub; ++m) {
      mbar_init(&vfull[m], 128);
      mbar_init(&accf[m], 1);
      mbar_init(&acce[m], kEpiWarps);
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
    if (lane == 0 && nseg > 0) {
      tma_prefetch_desc(&tw);
      int wt = 0;
      bool ok = true;
      for (int q = 0; ok && q < nseg; ++q) {
        const Seg sg = seg_at(lo, hi, nwt, q);
        int b, h, blk;
        unit_coords(a, sg.u, b, h, blk);
        for (int j = sg.j0; j < sg.j1; ++j, ++wt) {
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
      ring_tail(wempty, kWStages, wt, &s_abort, a.wc);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0 && nseg > 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kNT);
      const uint64_t vdesc = sdesc_kmajor_sw128(smem_u32(sV));
      bool ok = true;
      int wt = 0;   // W tiles (= rounds per accumulator) so far
      for (int q = 0; ok && q < nseg; ++q) {
        const Seg sg = seg_at(lo, hi, nwt, q);
        for (int j = sg.j0; ok && j < sg.j1; ++j, ++wt) {
          const int s = wt % kWStages, us = wt / kWStages;
          const uint64_t wdesc = sdesc_kmajor_sw128(smem_u32(sW + s * kWTile));
#pragma unroll
          for (int m = 0; m < kMsub; ++m) {
            const int uses = wt;   // earlier rounds on accumulator m
            if ((m == 0 && !mbar_wait(&wfull[s], us & 1, &s_abort, a.wc)) ||
                (j == sg.j0 && !mbar_wait(&vfull[m], q & 1, &s_abort, a.wc)) ||
                !mbar_wait(&acce[m], (uses & 1) ^ 1, &s_abort, a.wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              // descriptor start addresses advance in 16-byte units
              const uint32_t aoff = (m * kVSub + (k >> 2) * (128 * 128) + (k & 3) * 32) >> 4;
              const uint32_t boff = ((k >> 2) * (kNT * 128) + (k & 3) * 32) >> 4;
              umma_bf16(tbase + m * kAccCols, vdesc + aoff, wdesc + boff, idesc, k > 0 ? 1u : 0u);
            }
            umma_commit(&accf[m]);
          }
          if (ok) umma_commit(&wempty[s]);
        }
      }
      umma_commit(&done_bar);
      mbar_drain(&done_bar, 0, status);
    }
  } else {
    // epilogue: warp (q4, hf) reads TMEM lane quadrant q4, columns [hf*128, hf*128 + 128)
    // of every round, and owns the value row of token q4*32 + lane of subtile hf
    const int q4 = warp & 3, hf = warp >> 2;
    const int vr = q4 * 32 + lane;
    uint8_t* my_sub = sV + hf * kVSub;
    uint4 row[16];
    if (nseg > 0) {
      load_v_row(a, seg_at(lo, hi, nwt, 0).u, hf, vr, row);
      store_v_row(my_sub, vr, row);
      fence_proxy_async_smem();
      mbar_arrive(&vfull[hf]);
      if (nseg > 1) load_v_row(a, seg_at(lo, hi, nwt, 1).u, hf, vr, row);
    }
    bool ok = true;
    int wt = 0;
    for (int q = 0; q < nseg; ++q) {
      const Seg sg = seg_at(lo, hi, nwt, q);
      const int u = sg.u;
      float sm[kMsub][2];
#pragma unroll
      for (int m = 0; m < kMsub; ++m) sm[m][0] = sm[m][1] = 0.f;
      for (int j = sg.j0; j < sg.j1; ++j, ++wt) {
#pragma unroll
        for (int m = 0; m < kMsub; ++m) {
          if (!ok) continue;   // after an abort: fall through to the segment's vote
          const int uses = wt;
          const bool w = mbar_wait(&accf[m], uses & 1, &s_abort, a.wc);
          ok = __all_sync(0xffffffffu, w);
          if (!ok) continue;
          tc_fence_after();
          const uint32_t taddr = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + m * kAccCols + hf * kEpiCols;
          float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
          for (int c0 = 0; c0 < kEpiCols; c0 += 64) {
            float v[64];
            tmem_ld32(taddr + c0, v);
            tmem_ld32(taddr + c0 + 32, v + 32);
            tmem_ld_wait();
            if (c0 + 64 == kEpiCols) {
              // every column of this round is in registers: release the accumulator
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acce[m]);
            }
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
              p0 += fabsf(v[i + 0]);
              p1 += fabsf(v[i + 1]);
              p2 += fabsf(v[i + 2]);
              p3 += fabsf(v[i + 3]);
            }
          }
          sm[m][0] += p0 + p1;
          sm[m][1] += p2 + p3;
          if (j == sg.j1 - 1 && m == hf && q + 1 < nseg) {
            // every UMMA reading subtile hf of this segment has completed: refill it with
            // the next segment's rows, then fetch the rows of the segment after that
            store_v_row(my_sub, vr, row);
            fence_proxy_async_smem();
            mbar_arrive(&vfull[hf]);
            if (q + 2 < nseg) load_v_row(a, seg_at(lo, hi, nwt, q + 2).u, hf, vr, row);
          }
        }
      }
      // the two column halves of every token meet in shared memory; the barrier also
      // tells all eight warps whether any of them gave up
      if (hf == 1 && ok) {
#pragma unroll
        for (int m = 0; m < kMsub; ++m) s_half[m][vr] = sm[m][0] + sm[m][1];
      }
      if (epi_vote_any(!ok)) break;
      if (hf == 0) {
        int b, h, blk;
        unit_coords(a, u, b, h, blk);
        const int n = a.rq.n[b];
#pragma unroll
        for (int m = 0; m < kMsub; ++m) {
          const int tok = blk * kTokBlock + m * 128 + vr;
          if (tok < n) atomicAdd(a.nu + a.rq.soff[b] + static_cast<size_t>(h) * n + tok, (sm[m][0] + sm[m][1]) + s_half[m][vr]);
        }
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");   // s_half is read before the next unit writes it
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
                            int wo_mode, float* __restrict__ nu, long long nu_count) {
  const long long total = static_cast<long long>(H) * D * 16;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // nu is accumulated atomically by vnorm_kernel, which runs next on the stream
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nu_count; i += stride) nu[i] = 0.f;
  const long long row_len = static_cast<long long>(H) * G * kHeadDim;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total; t += stride) {
    const int c8 = static_cast<int>(t % 16);
    const long long hj = t / 16;
    const int j = static_cast<int>(hj % D);
    const int h = static_cast<int>(hj / D);
    const uint16_t* src = w_o + j * row_len + static_cast<long long>(h) * G * kHeadDim + c8 * 8;
    if (wo_mode == 0) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      // the loads of four slices are issued together, then summed in slice order
      for (int g0 = 0; g0 < G; g0 += 4) {
        uint4 p[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          p[u] = g0 + u < G ? __ldg(reinterpret_cast<const uint4*>(src + (g0 + u) * kHeadDim)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (g0 + u >= G) break;
          const uint32_t w[4] = {p[u].x, p[u].y, p[u].z, p[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] += __uint_as_float(w[i] << 16);
            acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
          }
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

cudaError_t launch_wbar(const uint16_t* w_o, uint16_t* wbar, int H, int G, int D, int wo_mode, float* nu,
                        long long nu_count, cudaStream_t st) {
  const long long total = static_cast<long long>(H) * D * 16;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  wbar_kernel<<<static_cast<unsigned>(blocks < 65535 * 8 ? blocks : 65535 * 8), threads, 0, st>>>(w_o, wbar, H, G, D,
                                                                                                  wo_mode, nu, nu_count);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_vnorm(const VnormArgs& a, const CUtensorMap& tw, cudaStream_t st) {
  if (a.units_total <= 0) return cudaSuccess;
  const size_t smem = 1024 + kVTile + kWStages * kWTile;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(vnorm_kernel), smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (a.grid_cap > 0 && a.grid_cap < sms) sms = a.grid_cap;
  const int grid = a.units_total < sms ? a.units_total : sms;
  vnorm_kernel<<<grid, kThreads, smem, st>>>(tw, a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
