// C-ABI host layer of libkvsel: argument validation, the per-call plan (budgets, key
// chunking, workspace layout), TMA tensor maps, and the launches of the scoring,
// selection and compaction kernels on the caller's stream.  Nothing here allocates
// device or host memory.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "../../include/kvsel.h"
#include "internal.cuh"

using namespace kvsel;

namespace kvsel {
cudaError_t ensure_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& cur = done[std::make_pair(func, dev)];
  if (cur >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) cur = bytes;
  if (e == cudaSuccess && func != nullptr) {
    // non-portable cluster sizes (16 CTAs) are allowed for every kernel that asks
    cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaGetLastError();
  }
  return e;
}

std::atomic<unsigned long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace kvsel

namespace {

constexpr unsigned long long kDefaultWaitCycles = 2000000000ull;   // ~1 s at the boost clock

thread_local void* const* t_stage_events = nullptr;

// Brackets one launch with the caller's diagnostic events (kvsel_set_stage_events).
struct StageScope {
  int stage;
  cudaStream_t st;
  StageScope(int s, cudaStream_t stream) : stage(s), st(stream) { rec(2 * stage); }
  ~StageScope() { rec(2 * stage + 1); }
  void rec(int i) const {
    if (!t_stage_events || !t_stage_events[i]) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(st, &cs);
    // under stream capture the record must become an external event node to time replays
    if (cs == cudaStreamCaptureStatusActive)
      cudaEventRecordWithFlags(static_cast<cudaEvent_t>(t_stage_events[i]), st, cudaEventRecordExternal);
    else
      cudaEventRecord(static_cast<cudaEvent_t>(t_stage_events[i]), st);
  }
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Plan {
  int B = 0, H = 0, G = 0, D = 0, W = 0, R = 0, R_pad = 0, n_max = 0, mt = 1, Dw = 0;
  bool qa = false;     // query-agnostic scoring (window == 0)
  ReqTable rq{};
  long long n_scores = 0;
  long long n_kept = 0;
  int budget[kMaxBatch]{}, budget1[kMaxBatch]{}, floor_h[kMaxBatch]{}, nforced[kMaxBatch]{};
  long long seg_out[kMaxBatch + 1]{};
  int max_count = 0;
  ChunkTable ck{};
  int units_total = 0, unit_base[kMaxBatch + 1]{}, blocks_per_head[kMaxBatch]{};
  bool l2 = false;     // value norm through the Gram matrix (KVSEL_NORM_L2)
  bool anchor = false; // AnchorKV anchors (KVSEL_BUDGET_ANCHOR)
  int ap_units = 0, ap_unit_base[kMaxBatch + 1]{}, ap_tiles[kMaxBatch]{};   // (b, h, side, 128-token tile)
  size_t ws_ainv = 0;  // anchors: 1/|a| of the K and V anchor rows
  int g_units = 0, g_unit_base[kMaxBatch + 1]{}, g_blocks_per_head[kMaxBatch]{};   // 128-token tiles
  int num_sms = 0;
  size_t ws_part = 0, ws_sraw = 0, ws_nu = 0, ws_wbar = 0, ws_total = 0;
  size_t ws_c2 = 0, ws_tmax = 0;   // query-agnostic scoring
  size_t ws_gpart = 0, ws_gam = 0;  // L2 value norm: Gram partials and Gamma hi/lo
  int qa_row_blocks = 0, qa_key_blocks = 0, qa_row_splits = 0;
  unsigned long long wait_limit = kDefaultWaitCycles;   // cycles one device-side wait may spin
  bool prepared = false;   // w_o is kvsel_prepare_w_o's output
  size_t prep_bytes = 0;   // its size
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVSEL_ECUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVSEL_ECUDA;
  return KVSEL_OK;
}

// Everything derived from the parameters alone (no pointers).  `need_device` asks for
// the SM count, which sets the key chunking and therefore the workspace size.
int make_plan(const kvsel_params* p, Plan& pl, bool need_device) {
  if (!p) return KVSEL_EINVAL;
  if (p->head_dim != kHeadDim) return KVSEL_EUNSUPPORTED;
  if (p->h_kv < 1 || p->h_kv > 64 || p->group < 1 || p->batch < 1 || p->batch > kMaxBatch) return KVSEL_EINVAL;
  if (p->reduce < 0 || p->reduce > 3 || p->pool < 0 || p->pool > 2) return KVSEL_EINVAL;
  if (p->reduce == KVSEL_REDUCE_MAX_LOGIT && p->window != 0) return KVSEL_EUNSUPPORTED;   // query-agnostic only
  if (p->pool != KVSEL_POOL_NONE && (p->pool_kernel < 1 || (p->pool_kernel & 1) == 0)) return KVSEL_EINVAL;
  if (p->budget_mode != KVSEL_BUDGET_PER_HEAD && p->budget_mode != KVSEL_BUDGET_PER_LAYER &&
      p->budget_mode != KVSEL_BUDGET_ANCHOR)
    return KVSEL_EINVAL;
  pl.anchor = p->budget_mode == KVSEL_BUDGET_ANCHOR;
  pl.wait_limit = p->wait_cycles ? p->wait_cycles : kDefaultWaitCycles;
  if (p->sm_budget < 0 || p->concurrent < 0 || p->concurrent > 1) return KVSEL_EINVAL;
  if (pl.anchor && !(p->alpha >= 0.f && p->alpha <= 1.f)) return KVSEL_EINVAL;
  if (!(p->budget_ratio >= 0.0 && p->budget_ratio <= 1.0) || !(p->floor_ratio >= 0.0 && p->floor_ratio <= 1.0))
    return KVSEL_EINVAL;
  if (p->n_sink < 0 || p->n_recent < 0 || p->window < 0 || !(p->scale >= 0.f) || std::isinf(p->scale))
    return KVSEL_EINVAL;
  if (p->value_aware) {
    if (p->wo_mode != KVSEL_WO_GROUP_SUM && p->wo_mode != KVSEL_WO_PER_HEAD) return KVSEL_EINVAL;
    if (p->d_model < 128 || p->d_model % 128 != 0) return KVSEL_EUNSUPPORTED;
    if (!(p->alpha >= 0.f && p->alpha <= 1.f) || !(p->eps >= 0.f)) return KVSEL_EINVAL;
    if (p->budget_mode == KVSEL_BUDGET_ANCHOR) return KVSEL_EUNSUPPORTED;
    if (p->value_norm != KVSEL_NORM_L1 && p->value_norm != KVSEL_NORM_L2) return KVSEL_EINVAL;
    // the Gram identity holds for one projection per token: the group-sum reading only
    if (p->value_norm == KVSEL_NORM_L2 && p->wo_mode != KVSEL_WO_GROUP_SUM) return KVSEL_EUNSUPPORTED;
    if (p->value_norm == KVSEL_NORM_L2 && p->group > 8) return KVSEL_EUNSUPPORTED;   // Gram staging fits G <= 8
    pl.l2 = p->value_norm == KVSEL_NORM_L2;
    if (p->w_o_prepared != 0 && p->w_o_prepared != 1) return KVSEL_EINVAL;
    pl.prepared = p->w_o_prepared == 1;
  }
  pl.B = p->batch;
  pl.H = p->h_kv;
  pl.G = p->group;
  pl.D = p->d_model;
  pl.W = p->window;
  pl.qa = (p->window == 0);
  pl.rq.B = pl.B;
  pl.rq.H = pl.H;
  long long so = 0;
  for (int b = 0; b < pl.B; ++b) {
    const int n = p->n_ctx_per_req ? p->n_ctx_per_req[b] : p->n_ctx;
    if (n < 0) return KVSEL_EINVAL;
    pl.rq.n[b] = n;
    pl.rq.soff[b] = so;
    so += static_cast<long long>(pl.H) * n;
    pl.n_max = n > pl.n_max ? n : pl.n_max;
  }
  pl.n_scores = so;
  if (so > (1ll << 31) - 1) return KVSEL_EUNSUPPORTED;
  if (pl.qa) {
    // KVzip's query-agnostic score: one request, all G*n positions as queries, no causal
    // mask, max over queries and group heads
    if (pl.B != 1 || p->causal || (p->reduce != KVSEL_REDUCE_MAX && p->reduce != KVSEL_REDUCE_MAX_LOGIT) ||
        p->value_aware || p->q_chunk < 0)
      return KVSEL_EUNSUPPORTED;
    if (static_cast<long long>(pl.G) * pl.n_max > (1ll << 30)) return KVSEL_EUNSUPPORTED;
    pl.R = 0;
    pl.R_pad = 64;
  } else {
    for (int b = 0; b < pl.B; ++b)
      if (pl.rq.n[b] > 0 && pl.W > pl.rq.n[b]) return KVSEL_EINVAL;
    pl.R = pl.G * pl.W;
    if (pl.R > 512 || pl.R % 32 != 0) return KVSEL_EUNSUPPORTED;
    pl.R_pad = (pl.R + 63) / 64 * 64;
    pl.mt = pl.R <= 128 ? 1 : (pl.R <= 256 ? 2 : 4);
  }
  pl.Dw = p->value_aware ? (p->wo_mode == KVSEL_WO_PER_HEAD ? pl.G * pl.D : pl.D) : 0;

  // budgets and output layout
  long long out = 0;
  for (int b = 0; b < pl.B; ++b) {
    const int n = pl.rq.n[b];
    const int nf = static_cast<int>(std::min<long long>(n, static_cast<long long>(p->n_sink) + p->n_recent));
    pl.nforced[b] = nf;
    pl.seg_out[b] = out;
    if (pl.anchor) {
      // AnchorKV: k = floor(ratio * n) anchors, at least the forced window, at most n;
      // floor(rho * (k - |F|)) of the free slots by score, the rest by the random keys
      long long k = static_cast<long long>(std::floor(p->budget_ratio * static_cast<double>(n)));
      k = std::min<long long>(std::max<long long>(k, nf), n);
      pl.budget[b] = static_cast<int>(k);
      pl.budget1[b] =
          nf + static_cast<int>(std::floor(static_cast<double>(p->alpha) * static_cast<double>(k - nf)));
      out += static_cast<long long>(pl.H) * k;
      pl.max_count = std::max(pl.max_count, static_cast<int>(k));
    } else if (p->budget_mode == KVSEL_BUDGET_PER_HEAD) {
      const long long B = static_cast<long long>(std::floor(p->budget_ratio * static_cast<double>(n)));
      if (B < nf || B > n) return KVSEL_EBUDGET;
      pl.budget[b] = static_cast<int>(B);
      long long b1 = static_cast<long long>(std::floor(static_cast<double>(p->alpha) * static_cast<double>(B)));
      if (b1 < nf) b1 = nf;
      pl.budget1[b] = static_cast<int>(b1);
      out += static_cast<long long>(pl.H) * B;
      pl.max_count = std::max(pl.max_count, static_cast<int>(B));
    } else {
      const long long BL =
          static_cast<long long>(std::floor(p->budget_ratio * static_cast<double>(n) * static_cast<double>(pl.H)));
      const long long fl = static_cast<long long>(std::floor(p->floor_ratio * static_cast<double>(n)));
      const long long fh = std::min<long long>(n, std::max<long long>(fl, nf));
      if (BL < fh * pl.H || BL > static_cast<long long>(n) * pl.H) return KVSEL_EBUDGET;
      pl.budget[b] = static_cast<int>(BL);
      pl.floor_h[b] = static_cast<int>(fl);
      out += BL;
      pl.max_count = std::max(pl.max_count, static_cast<int>(std::min<long long>(BL, n)));
    }
  }
  pl.seg_out[pl.B] = out;
  pl.n_kept = out;

  if (!need_device) return KVSEL_OK;
  int rc = device_sms(&pl.num_sms);
  if (rc) return rc;
  if (p->sm_budget > 0 && p->sm_budget < pl.num_sms) pl.num_sms = p->sm_budget;

  // key chunks: about one chunk per SM over all (request, head) pairs
  long long t256 = 0;
  for (int b = 0; b < pl.B; ++b) t256 += static_cast<long long>(pl.H) * ((pl.rq.n[b] + 255) / 256);
  long long tpc = (t256 + pl.num_sms - 1) / std::max(pl.num_sms, 1);
  if (tpc < 1) tpc = 1;
  // at most 64 chunks per head (the pass-2 merge reads a row's partials in one sweep)
  const long long min_tpc = (static_cast<long long>((pl.n_max + 255) / 256) + 63) / 64;
  if (tpc < min_tpc) tpc = min_tpc;
  pl.ck.chunk_len = static_cast<int>(256 * tpc);
  int cb = 0, pb = 0;
  for (int b = 0; b < pl.B; ++b) {
    pl.ck.base[b] = cb;
    pl.ck.pbase[b] = pb;
    pl.ck.per_head[b] = (pl.rq.n[b] + pl.ck.chunk_len - 1) / pl.ck.chunk_len;
    cb += pl.H * pl.ck.per_head[b];
    pb += pl.H * chunk_pad(pl.ck.per_head[b]);
  }
  pl.ck.base[pl.B] = cb;
  pl.ck.pbase[pl.B] = pb;
  pl.ck.total = cb;

  const int tb = vnorm_token_block();
  int ub = 0;
  for (int b = 0; b < pl.B; ++b) {
    pl.unit_base[b] = ub;
    pl.blocks_per_head[b] = (pl.rq.n[b] + tb - 1) / tb;
    ub += pl.H * pl.blocks_per_head[b];
  }
  pl.unit_base[pl.B] = ub;
  pl.units_total = p->value_aware ? ub : 0;
  int gu = 0;
  for (int b = 0; b < pl.B; ++b) {
    pl.g_unit_base[b] = gu;
    pl.g_blocks_per_head[b] = (pl.rq.n[b] + 127) / 128;
    gu += pl.H * pl.g_blocks_per_head[b];
  }
  pl.g_unit_base[pl.B] = gu;
  pl.g_units = pl.l2 ? gu : 0;
  int au = 0;
  for (int b = 0; b < pl.B; ++b) {
    pl.ap_unit_base[b] = au;
    pl.ap_tiles[b] = (pl.rq.n[b] + 127) / 128;
    au += pl.H * 2 * pl.ap_tiles[b];
  }
  pl.ap_unit_base[pl.B] = au;
  pl.ap_units = pl.anchor ? au : 0;

  size_t off = kStatusBytes + kCounterBytes;
  if (pl.qa) {
    const int n = pl.rq.n[0];
    const long long GN = static_cast<long long>(pl.G) * n;
    const int br = qa_block_rows();
    pl.qa_row_blocks = static_cast<int>((GN + br - 1) / br);
    pl.qa_key_blocks = (n + qa_key_block() - 1) / qa_key_block();
    // query-row slices per key block: at least eight CTAs per SM in all, and a whole
    // number of waves (one CTA per SM) to within 3% where a slice count up to 64 gives one
    const long long want = 8ll * pl.num_sms;
    const long long base = static_cast<long long>(pl.H) * std::max(pl.qa_key_blocks, 1);
    const int s0 = static_cast<int>(std::min<long long>(64, std::max<long long>(1, (want + base - 1) / base)));
    int best_s = s0;
    double best_eff = 0.0;
    for (int sp = s0; sp <= 64; ++sp) {
      const long long ctas = base * sp;
      const long long waves = (ctas + pl.num_sms - 1) / pl.num_sms;
      const double eff = static_cast<double>(ctas) / static_cast<double>(waves * pl.num_sms);
      if (eff > best_eff + 1e-9) {
        best_eff = eff;
        best_s = sp;
      }
      if (eff >= 0.97) break;
    }
    pl.qa_row_splits = best_s;
    pl.ws_c2 = off;
    off = align256(off + static_cast<size_t>(pl.H) * GN * sizeof(float));
    pl.ws_tmax = off;
    off = align256(off + static_cast<size_t>(pl.n_scores) * sizeof(uint32_t));
    pl.ws_sraw = off;
    off = align256(off + static_cast<size_t>(pl.n_scores) * sizeof(float));
    if (pl.anchor) {
      pl.ws_ainv = off;
      off = align256(off + 2 * static_cast<size_t>(pl.n_kept) * sizeof(float));
    }
    pl.ws_total = off;
    return KVSEL_OK;
  }
  pl.ws_part = off;
  off = align256(off + static_cast<size_t>(pl.ck.pbase[pl.B]) * 2 * pl.R_pad * sizeof(float));
  pl.ws_sraw = off;
  off = align256(off + static_cast<size_t>(pl.n_scores) * sizeof(float));
  if (p->value_aware) {
    pl.ws_nu = off;
    off = align256(off + static_cast<size_t>(pl.n_scores) * sizeof(float));
    pl.prep_bytes = pl.l2 ? static_cast<size_t>(pl.H) * 2 * kHeadDim * kHeadDim * 2
                          : static_cast<size_t>(pl.H) * pl.Dw * kHeadDim * 2;
    if (!pl.l2 && !pl.prepared) {
      pl.ws_wbar = off;   // W_h (the L1 path; the L2 path never materialises it)
      off = align256(off + pl.prep_bytes);
    }
    if (pl.l2) {
      // the Gram partials (also what kvsel_prepare_w_o needs), and Gamma unless prepared
      pl.ws_gpart = off;
      off = align256(off + static_cast<size_t>(pl.H) * gram_slices(pl.Dw) * kHeadDim * kHeadDim * sizeof(float));
      if (!pl.prepared) {
        pl.ws_gam = off;
        off = align256(off + pl.prep_bytes);
      }
    }
  }
  if (pl.anchor) {
    pl.ws_ainv = off;
    off = align256(off + 2 * static_cast<size_t>(pl.n_kept) * sizeof(float));
  }
  pl.ws_total = off;
  return KVSEL_OK;
}

int check_kv(const kvsel_kv* kv, const Plan& pl, bool need_v) {
  if (!kv || !kv->k || (need_v && !kv->v)) return KVSEL_EINVAL;
  if (!aligned16(kv->k) || (kv->v && !aligned16(kv->v))) return KVSEL_EINVAL;
  if (kv->layout == KVSEL_LAYOUT_CONTIGUOUS) {
    if (kv->stride_tok < kHeadDim || kv->stride_head < 0 || kv->stride_req < 0) return KVSEL_EINVAL;
    if ((kv->stride_tok * 2) % 16 || (kv->stride_head * 2) % 16 || (kv->stride_req * 2) % 16) return KVSEL_EINVAL;
    if (pl.H > 1 && kv->stride_head == 0) return KVSEL_EINVAL;
    if (pl.B > 1 && kv->stride_req == 0) return KVSEL_EINVAL;
  } else if (kv->layout == KVSEL_LAYOUT_PAGED) {
    const int bs = kv->block_size;
    if (!kv->block_table || !(bs == 8 || bs == 16 || bs == 32 || bs == 64)) return KVSEL_EINVAL;
    if (kv->num_blocks < 1 || kv->max_blocks < (pl.n_max + bs - 1) / bs) return KVSEL_EINVAL;
  } else {
    return KVSEL_EINVAL;
  }
  return KVSEL_OK;
}

// The driver's tensor-map encoder, looked up through the runtime so that the library
// loads on machines without a driver (symbol checks) and links no libcuda.
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
            const cuuint32_t* box) {
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims,
                                            strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// K or V tiles of `rows` tokens.
bool kv_map(CUtensorMap* m, const void* base, const kvsel_kv* kv, const Plan& pl, int rows) {
  if (kv->layout == KVSEL_LAYOUT_CONTIGUOUS) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(std::max(pl.n_max, 1)),
                                static_cast<cuuint64_t>(pl.H), static_cast<cuuint64_t>(pl.B)};
    const long long sh = pl.H > 1 ? kv->stride_head : static_cast<long long>(std::max(pl.n_max, 1)) * kv->stride_tok;
    const long long sr = pl.B > 1 ? kv->stride_req : sh * pl.H;
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kv->stride_tok * 2), static_cast<cuuint64_t>(sh * 2),
                                   static_cast<cuuint64_t>(sr * 2)};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(rows), 1, 1};
    return encode(m, base, 4, dims, strides, box);
  }
  const int bs = kv->block_size;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(pl.H),
                              static_cast<cuuint64_t>(bs), static_cast<cuuint64_t>(kv->num_blocks)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHeadDim * 2), static_cast<cuuint64_t>(pl.H) * kHeadDim * 2,
                                 static_cast<cuuint64_t>(bs) * pl.H * kHeadDim * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(bs), 1};
  return encode(m, base, 4, dims, strides, box);
}

KvSource kv_source(const kvsel_kv* kv) {
  KvSource s{};
  s.paged = kv->layout == KVSEL_LAYOUT_PAGED;
  s.block_size = kv->block_size;
  s.max_blocks = kv->max_blocks;
  s.num_blocks = kv->num_blocks;
  s.block_table = kv->block_table;
  return s;
}

int launch_rc(cudaError_t e) { return e == cudaSuccess ? KVSEL_OK : KVSEL_ECUDA; }

int check_ws(const Plan& pl, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return KVSEL_EWORKSPACE;
  if (ws_bytes < pl.ws_total) return KVSEL_EWORKSPACE;
  return KVSEL_OK;
}

WaitCtl wait_ctl(const Plan& pl, void* ws) { return WaitCtl{pl.wait_limit, static_cast<int*>(ws)}; }

int do_score(const kvsel_params* p, const Plan& pl, const void* q, const kvsel_kv* kv, const void* w_o, float* s_attn,
             float* s_val, void* ws, cudaStream_t st, bool finalize = true) {
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* part = reinterpret_cast<float*>(wsb + pl.ws_part);
  float* s_raw = reinterpret_cast<float*>(wsb + pl.ws_sraw);
  if (pl.n_scores == 0) return KVSEL_OK;
  const float scale = p->scale > 0.f ? p->scale : 1.f / std::sqrt(static_cast<float>(kHeadDim));
  if (pl.qa) {
    const int n = pl.rq.n[0];
    CUtensorMap tq, tq2, tk128;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(pl.H) * pl.G * n};
    const cuuint64_t strides[1] = {kHeadDim * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t box2[2] = {64, static_cast<cuuint32_t>(qa_query_tile())};   // pass 2: one tile per column half
    if (!encode(&tq, q, 2, dims, strides, box) || !encode(&tq2, q, 2, dims, strides, box2)) return KVSEL_EINVAL;
    if (!kv_map(&tk128, kv->k, kv, pl, 128)) return KVSEL_EINVAL;
    QaArgs a{};
    a.H = pl.H;
    a.n = n;
    a.GN = pl.G * n;
    a.row_blocks = pl.qa_row_blocks;
    a.key_blocks = pl.qa_key_blocks;
    a.row_splits = pl.qa_row_splits;
    a.logit = p->reduce == KVSEL_REDUCE_MAX_LOGIT ? 1 : 0;
    a.s2 = a.logit ? scale : scale * 1.4426950408889634f;
    a.c2 = reinterpret_cast<float*>(wsb + pl.ws_c2);
    a.tmax = reinterpret_cast<uint32_t*>(wsb + pl.ws_tmax);
    a.s_raw = s_raw;
    a.wc = wait_ctl(pl, ws);
    int rc;
    if (!a.logit) {
      StageScope sc(KVSEL_STAGE_ROWSTATS, st);
      rc = launch_rc(launch_qa_rowlse(a, tq, tk128, st));
      if (rc) return rc;
    }
    {
      StageScope sc(KVSEL_STAGE_KEYSUM, st);
      rc = launch_rc(launch_qa_keymax(a, tq2, tk128, st));
    }
    if (rc) return rc;
    StageScope sc(KVSEL_STAGE_FINALIZE, st);
    if (!finalize) return KVSEL_OK;   // pooling happens inside the selection (kvsel_run_layer)
    return launch_rc(launch_finalize(pl.rq, s_raw, nullptr, s_attn, nullptr, p->pool, p->pool_kernel, p->eps, st));
  }

  CUtensorMap tq, tk1, tk2;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(pl.B) * pl.H * pl.R};
    const cuuint64_t strides[1] = {kHeadDim * 2};
    const cuuint32_t box[2] = {64, 32};
    if (!encode(&tq, q, 2, dims, strides, box)) return KVSEL_EINVAL;
  }
  const int nt1 = pl.mt == 4 ? 64 : 128;
  if (!kv_map(&tk1, kv->k, kv, pl, kv->layout == KVSEL_LAYOUT_PAGED ? 0 : nt1)) return KVSEL_EINVAL;
  if (!kv_map(&tk2, kv->k, kv, pl, kv->layout == KVSEL_LAYOUT_PAGED ? 0 : 128)) return KVSEL_EINVAL;

  WinScoreArgs a{};
  a.rq = pl.rq;
  a.ck = pl.ck;
  a.src = kv_source(kv);
  a.G = pl.G;
  a.W = pl.W;
  a.R = pl.R;
  a.R_pad = pl.R_pad;
  a.causal = p->causal ? 1 : 0;
  a.reduce = p->reduce;
  a.s2 = scale * 1.4426950408889634f;
  a.part = part;
  a.s_raw = s_raw;
  // the L1 value norms are accumulated atomically: the fused launch zeroes them on the way
  a.nu_zero = (p->value_aware && !pl.l2) ? reinterpret_cast<float*>(wsb + pl.ws_nu) : nullptr;
  a.wc = wait_ctl(pl, ws);
  int rc;
  cudaError_t fe = cudaErrorNotSupported;
  if (pl.mt <= 2 && !p->concurrent) {
    // both passes in one cooperative launch when every chunk fits on the device at once
    // (not when other work may hold SMs: the launch's CTAs wait for each other)
    StageScope sc(KVSEL_STAGE_ROWSTATS, st);
    fe = launch_win_fused(a, tq, tk2, reinterpret_cast<unsigned int*>(wsb + kStatusBytes), st);
    if (fe != cudaSuccess && fe != cudaErrorNotSupported) return KVSEL_ECUDA;
  }
  if (fe == cudaSuccess) StageScope sc(KVSEL_STAGE_KEYSUM, st);   // pass 2 ran inside the fused launch
  if (fe == cudaErrorNotSupported) {
    {
      StageScope sc(KVSEL_STAGE_ROWSTATS, st);
      rc = launch_rc(launch_win_rowstats(a, tq, tk1, pl.mt, st));
    }
    if (rc) return rc;
    {
      StageScope sc(KVSEL_STAGE_KEYSUM, st);
      rc = launch_rc(launch_win_keysum(a, tq, tk2, st));
    }
    if (rc) return rc;
  }

  float* nu = nullptr;
  if (p->value_aware && pl.l2) {
    // nu = ||W_h v||_2 = sqrt(v^T Gamma_h v) with Gamma_h = W_h^T W_h (d x d)
    nu = reinterpret_cast<float*>(wsb + pl.ws_nu);
    float* gpart = reinterpret_cast<float*>(wsb + pl.ws_gpart);
    uint16_t* gam = pl.prepared ? static_cast<uint16_t*>(const_cast<void*>(w_o))
                                : reinterpret_cast<uint16_t*>(wsb + pl.ws_gam);
    CUtensorMap two, tg, tv;
    if (!pl.prepared) {
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(pl.H) * pl.G * kHeadDim, static_cast<cuuint64_t>(pl.D)};
      const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pl.H) * pl.G * kHeadDim * 2};
      const cuuint32_t box[2] = {64, 64};
      if (!encode(&two, w_o, 2, dims, strides, box)) return KVSEL_EINVAL;
    }
    {
      const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(pl.H) * 2 * kHeadDim};
      const cuuint64_t strides[1] = {kHeadDim * 2};
      const cuuint32_t box[2] = {64, 128};
      if (!encode(&tg, gam, 2, dims, strides, box)) return KVSEL_EINVAL;
    }
    if (!kv_map(&tv, kv->v, kv, pl, kv->layout == KVSEL_LAYOUT_PAGED ? 0 : 128)) return KVSEL_EINVAL;
    if (!pl.prepared) {
      StageScope sc(KVSEL_STAGE_WBAR, st);
      rc = launch_rc(launch_value_gram(two, gpart, gam, pl.H, pl.G, pl.D, wait_ctl(pl, ws), st));
    }
    if (rc) return rc;
    VgramArgs v{};
    v.rq = pl.rq;
    v.src = kv_source(kv);
    v.units_total = pl.g_units;
    for (int b = 0; b <= pl.B; ++b) v.unit_base[b] = pl.g_unit_base[b];
    for (int b = 0; b < pl.B; ++b) v.blocks_per_head[b] = pl.g_blocks_per_head[b];
    v.nu = nu;
    v.grid_cap = pl.num_sms;
    v.wc = wait_ctl(pl, ws);
    {
      StageScope sc(KVSEL_STAGE_VNORM, st);
      rc = launch_rc(launch_vgram(v, tv, tg, st));
    }
    if (rc) return rc;
  } else if (p->value_aware) {
    nu = reinterpret_cast<float*>(wsb + pl.ws_nu);
    uint16_t* wbar = pl.prepared ? static_cast<uint16_t*>(const_cast<void*>(w_o))
                                 : reinterpret_cast<uint16_t*>(wsb + pl.ws_wbar);
    if (!pl.prepared || fe != cudaSuccess) {
      StageScope sc(KVSEL_STAGE_WBAR, st);
      // W_h (unless prepared) and the zeroed nu that the value-norm kernel accumulates into
      // (already zeroed by the fused scoring launch when that ran)
      rc = pl.prepared ? launch_rc(cudaMemsetAsync(nu, 0, static_cast<size_t>(pl.n_scores) * sizeof(float), st))
                       : launch_rc(launch_wbar(static_cast<const uint16_t*>(w_o), wbar, pl.H, pl.G, pl.D, p->wo_mode,
                                               nu, fe == cudaSuccess ? 0 : pl.n_scores, st));
      if (rc) return rc;
    }
    CUtensorMap tw;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(pl.Dw),
                                static_cast<cuuint64_t>(pl.H)};
    const cuuint64_t strides[2] = {kHeadDim * 2, static_cast<cuuint64_t>(pl.Dw) * kHeadDim * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(vnorm_w_tile_rows()), 1};
    if (!encode(&tw, wbar, 3, dims, strides, box)) return KVSEL_EINVAL;
    VnormArgs v{};
    v.rq = pl.rq;
    v.src = kv_source(kv);
    v.v = static_cast<const uint16_t*>(kv->v);
    v.stride_req = kv->stride_req;
    v.stride_head = kv->stride_head;
    v.stride_tok = kv->stride_tok;
    v.D = pl.D;
    v.Dw = pl.Dw;
    v.units_total = pl.units_total;
    for (int b = 0; b <= pl.B; ++b) v.unit_base[b] = pl.unit_base[b];
    for (int b = 0; b < pl.B; ++b) v.blocks_per_head[b] = pl.blocks_per_head[b];
    v.nu = nu;
    v.grid_cap = pl.num_sms;
    v.wc = wait_ctl(pl, ws);
    {
      StageScope sc(KVSEL_STAGE_VNORM, st);
      rc = launch_rc(launch_vnorm(v, tw, st));
    }
    if (rc) return rc;
  }
  StageScope sc(KVSEL_STAGE_FINALIZE, st);
  if (!finalize) return KVSEL_OK;   // pooling happens inside the selection (kvsel_run_layer)
  return launch_rc(launch_finalize(pl.rq, s_raw, nu, s_attn, p->value_aware ? s_val : nullptr, p->pool,
                                   p->pool_kernel, p->eps, st));
}

int do_select(const kvsel_params* p, const Plan& pl, const float* s_attn, const float* s_val, int32_t* idx,
              int32_t* counts, int64_t* offsets, cudaStream_t st, const float* raw = nullptr,
              const float* nu = nullptr, float* out_attn = nullptr, float* out_val = nullptr) {
  SelectArgs a{};
  a.raw = raw;
  a.nu = nu;
  a.out_attn = out_attn;
  a.out_val = out_val;
  a.pool = p->pool;
  a.pool_kernel = p->pool_kernel;
  a.eps = p->eps;
  a.rq = pl.rq;
  a.mode = p->budget_mode;
  // two stages: value-aware (CriticalKV Algorithm 1), or anchors (AnchorKV §3.2: the
  // second stage ranks by the caller's random keys, passed as s_val)
  a.two_stage = (p->value_aware || pl.anchor) ? 1 : 0;
  a.alpha = p->alpha;
  a.n_sink = p->n_sink;
  a.n_recent = p->n_recent;
  for (int b = 0; b < pl.B; ++b) {
    a.budget[b] = pl.budget[b];
    a.budget1[b] = pl.budget1[b];
    a.floor_h[b] = pl.floor_h[b];
    a.seg_out[b] = pl.seg_out[b];
  }
  a.s1 = s_attn;
  a.s2 = s_val;
  a.idx = idx;
  a.counts = counts;
  a.offsets = offsets;
  const int max_len = p->budget_mode == KVSEL_BUDGET_PER_LAYER ? pl.H * pl.n_max : pl.n_max;
  int cap = 0;
  const int segs = p->budget_mode == KVSEL_BUDGET_PER_LAYER ? pl.B : pl.B * pl.H;
  // overlapping calls: 4-CTA clusters, or 2 when four per segment would exceed the SMs the
  // call is sized for (many calls in flight)
  const auto min_cs = [&](int nseg) {
    if (!p->concurrent) return 0;
    return (p->sm_budget > 0 && 4ll * nseg > p->sm_budget) ? 2 : 4;
  };
  const int cs = select_cluster_size(std::max(max_len, 1), segs, min_cs(segs), &cap);
  if (cs < 0) return KVSEL_EUNSUPPORTED;
  StageScope sc(KVSEL_STAGE_SELECT, st);
  if (p->budget_mode != KVSEL_BUDGET_PER_LAYER || !p->value_aware) return launch_rc(launch_select(a, cs, cap, st));
  // Value-aware selection under a per-layer budget (CriticalKV Algorithm 2, line 1 then
  // line 8): the layer-wide top of the pooled attention score sets each head's budget
  // (counts/offsets; its pooling also writes s_attn and s_val), then the two-stage
  // selection runs per head within that budget, reading the budgets on the device.
  a.two_stage = 0;
  int rc = launch_rc(launch_select(a, cs, cap, st));
  if (rc) return rc;
  SelectArgs h = a;
  h.mode = KVSEL_BUDGET_PER_HEAD;
  h.two_stage = 1;
  h.raw = nullptr;
  h.nu = nullptr;
  h.out_attn = nullptr;
  h.out_val = nullptr;
  h.s1 = out_attn ? out_attn : s_attn;
  h.s2 = out_val ? out_val : s_val;
  h.dev_counts = counts;
  h.dev_offsets = offsets;
  int cap2 = 0;
  const int cs2 = select_cluster_size(std::max(pl.n_max, 1), pl.B * pl.H, min_cs(pl.B * pl.H), &cap2);
  if (cs2 < 0) return KVSEL_EUNSUPPORTED;
  return launch_rc(launch_select(h, cs2, cap2, st));
}

int do_compact(const Plan& pl, const kvsel_kv* kv, const int32_t* idx, const int32_t* counts, const int64_t* offsets,
               void* k_out, void* v_out, void* ws, cudaStream_t st) {
  CompactArgs c{};
  c.rq = pl.rq;
  c.src = kv_source(kv);
  c.k = static_cast<const uint16_t*>(kv->k);
  c.v = static_cast<const uint16_t*>(kv->v);
  c.stride_req = kv->stride_req;
  c.stride_head = kv->stride_head;
  c.stride_tok = kv->stride_tok;
  c.idx = idx;
  c.counts = counts;
  c.offsets = offsets;
  c.k_out = static_cast<uint16_t*>(k_out);
  c.v_out = static_cast<uint16_t*>(v_out);
  c.n_kept = pl.n_kept;
  c.status = static_cast<int*>(ws);
  int sms = pl.num_sms;
  if (!sms && device_sms(&sms)) return KVSEL_ECUDA;
  StageScope sc(KVSEL_STAGE_COMPACT, st);
  return launch_rc(launch_compact(c, pl.max_count, sms, st));
}

// Workspace of kvsel_perturbation, after the status word and counters.
struct PerturbLayout {
  size_t keep = 0, nu = 0, stat_part = 0, stat = 0, e_part = 0, e = 0, y_part = 0, total = 0;
};

int perturb_plan(const kvsel_params* p, const Plan& pl, PerturbLayout& L) {
  if (pl.qa || pl.R > 128 || pl.R < 1 || pl.G > 16) return KVSEL_EUNSUPPORTED;
  if (p->d_model < 128 || p->d_model % 128 != 0) return KVSEL_EUNSUPPORTED;
  size_t off = kStatusBytes + kCounterBytes;
  L.keep = off;
  off = align256(off + static_cast<size_t>(pl.n_scores));
  L.nu = off;
  off = align256(off + static_cast<size_t>(pl.G) * pl.n_scores * sizeof(float));
  L.stat_part = off;
  off = align256(off + static_cast<size_t>(pl.ck.total) * 128 * 7 * sizeof(float));
  L.stat = off;
  off = align256(off + static_cast<size_t>(pl.B) * pl.H * 128 * 7 * sizeof(float));
  L.e_part = off;
  off = align256(off + static_cast<size_t>(pl.ck.total) * 128 * 128 * sizeof(float));
  L.e = off;
  off = align256(off + static_cast<size_t>(pl.B) * pl.H * 128 * 128 * sizeof(float));
  L.y_part = off;
  off = align256(off + static_cast<size_t>(pl.B) * pl.H * pl.G * perturb_slices(pl.D) * pl.W * sizeof(float));
  L.total = off;
  return KVSEL_OK;
}

int do_anchor_project(const Plan& pl, const kvsel_kv* kv, const void* anchor_k, const void* anchor_v,
                      const int32_t* idx, const int32_t* counts, const int64_t* offsets, int32_t* slot_k,
                      float* gamma_k, int32_t* slot_v, float* gamma_v, void* ws, cudaStream_t st) {
  if (pl.n_scores == 0) return KVSEL_OK;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* inv = reinterpret_cast<float*>(wsb + pl.ws_ainv);
  CUtensorMap tk, tv, tak, tav;
  const int rows = kv->layout == KVSEL_LAYOUT_PAGED ? 0 : 128;
  if (!kv_map(&tk, kv->k, kv, pl, rows) || !kv_map(&tv, kv->v, kv, pl, rows)) return KVSEL_EINVAL;
  const long long nr = std::max<long long>(pl.n_kept, 1);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(nr)};
  const cuuint64_t strides[1] = {kHeadDim * 2};
  const cuuint32_t box[2] = {64, 256};
  if (!encode(&tak, anchor_k, 2, dims, strides, box) || !encode(&tav, anchor_v, 2, dims, strides, box))
    return KVSEL_EINVAL;
  StageScope sc(KVSEL_STAGE_PROJECT, st);
  int rc = launch_rc(launch_anchor_norms(static_cast<const uint16_t*>(anchor_k), static_cast<const uint16_t*>(anchor_v),
                                         pl.n_kept, inv, st));
  if (rc) return rc;
  AnchorArgs a{};
  a.rq = pl.rq;
  a.src = kv_source(kv);
  a.units_total = pl.ap_units;
  for (int b = 0; b <= pl.B; ++b) a.unit_base[b] = pl.ap_unit_base[b];
  for (int b = 0; b < pl.B; ++b) a.tiles[b] = pl.ap_tiles[b];
  a.idx = idx;
  a.counts = counts;
  a.offsets = offsets;
  a.n_rows = pl.n_kept;
  a.inv = inv;
  a.slot[0] = slot_k;
  a.slot[1] = slot_v;
  a.gamma[0] = gamma_k;
  a.gamma[1] = gamma_v;
  a.wc = wait_ctl(pl, ws);
  return launch_rc(launch_anchor_project(a, tk, tv, tak, tav, st));
}

int check_anchor_args(const Plan& pl, const kvsel_kv* kv, const void* anchor_k, const void* anchor_v,
                      const int32_t* idx, const int32_t* counts, const int64_t* offsets, const int32_t* slot_k,
                      const float* gamma_k, const int32_t* slot_v, const float* gamma_v, void* ws, size_t ws_bytes) {
  if (!pl.anchor) return KVSEL_EINVAL;
  if (pl.max_count > anchor_max()) return KVSEL_EUNSUPPORTED;
  if (!anchor_k || !anchor_v || !aligned16(anchor_k) || !aligned16(anchor_v) || !idx || !counts || !offsets)
    return KVSEL_EINVAL;
  if (!slot_k || !gamma_k || !slot_v || !gamma_v) return KVSEL_EINVAL;
  int rc = check_kv(kv, pl, true);
  if (rc) return rc;
  return check_ws(pl, ws, ws_bytes);
}

}  // namespace

extern "C" {

int kvsel_anchor_project(const kvsel_params* p, const kvsel_kv* kv, const void* anchor_k, const void* anchor_v,
                         const int32_t* idx, const int32_t* counts, const int64_t* offsets, int32_t* slot_k,
                         float* gamma_k, int32_t* slot_v, float* gamma_v, void* ws, size_t ws_bytes, void* stream) {
  Plan pl;
  int rc = make_plan(p, pl, true);
  if (rc) return rc;
  if ((rc = check_anchor_args(pl, kv, anchor_k, anchor_v, idx, counts, offsets, slot_k, gamma_k, slot_v, gamma_v, ws,
                              ws_bytes)))
    return rc;
  return do_anchor_project(pl, kv, anchor_k, anchor_v, idx, counts, offsets, slot_k, gamma_k, slot_v, gamma_v, ws,
                           static_cast<cudaStream_t>(stream));
}

int kvsel_perturbation_workspace_size(const kvsel_params* p, size_t* bytes) {
  if (!bytes) return KVSEL_EINVAL;
  Plan pl;
  int rc = make_plan(p, pl, true);
  if (rc) return rc;
  PerturbLayout L;
  if ((rc = perturb_plan(p, pl, L))) return rc;
  *bytes = L.total;
  return KVSEL_OK;
}

int kvsel_perturbation(const kvsel_params* p, const void* q, const kvsel_kv* kv, const void* w_o, const int32_t* idx,
                       const int32_t* counts, const int64_t* offsets, float* out, void* ws, size_t ws_bytes,
                       void* stream) {
  Plan pl;
  int rc = make_plan(p, pl, true);
  if (rc) return rc;
  PerturbLayout L;
  if ((rc = perturb_plan(p, pl, L))) return rc;
  if (p->w_o_prepared) return KVSEL_EINVAL;   // the harness projects through W_O's own slices
  if (!q || !aligned16(q) || !w_o || !aligned16(w_o) || !idx || !counts || !offsets || !out) return KVSEL_EINVAL;
  if ((rc = check_kv(kv, pl, true))) return rc;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < L.total) return KVSEL_EWORKSPACE;
  if (pl.n_scores == 0) return KVSEL_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const float scale = p->scale > 0.f ? p->scale : 1.f / std::sqrt(static_cast<float>(kHeadDim));
  PerturbArgs a{};
  a.rq = pl.rq;
  a.ck = pl.ck;
  a.src = kv_source(kv);
  a.G = pl.G;
  a.W = pl.W;
  a.R = pl.R;
  a.causal = p->causal ? 1 : 0;
  a.s2 = scale * 1.4426950408889634f;
  a.D = pl.D;
  a.keep = wsb + L.keep;
  a.nu = reinterpret_cast<const float*>(wsb + L.nu);
  a.n_scores = pl.n_scores;
  a.stat_part = reinterpret_cast<float*>(wsb + L.stat_part);
  a.stat = reinterpret_cast<float*>(wsb + L.stat);
  a.e_part = reinterpret_cast<float*>(wsb + L.e_part);
  a.e = reinterpret_cast<float*>(wsb + L.e);
  a.y_part = reinterpret_cast<float*>(wsb + L.y_part);
  a.out = out;
  a.wc = wait_ctl(pl, ws);
  CUtensorMap tq, tk, tv;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(pl.B) * pl.H * pl.R};
    const cuuint64_t strides[1] = {kHeadDim * 2};
    const cuuint32_t box[2] = {64, 128};
    if (!encode(&tq, q, 2, dims, strides, box)) return KVSEL_EINVAL;
  }
  const int rows = kv->layout == KVSEL_LAYOUT_PAGED ? 0 : 128;
  if (!kv_map(&tk, kv->k, kv, pl, rows) || !kv_map(&tv, kv->v, kv, pl, rows)) return KVSEL_EINVAL;
  StageScope sc(KVSEL_STAGE_PERTURB, st);
  // kept positions -> byte mask
  if ((rc = launch_rc(cudaMemsetAsync(wsb + L.keep, 0, static_cast<size_t>(pl.n_scores), st)))) return rc;
  if ((rc = launch_rc(launch_perturb_mask(pl.rq, idx, counts, offsets, pl.n_max, wsb + L.keep, static_cast<int*>(ws),
                                          st))))
    return rc;
  // ||W_O^(h,g) v_i||_1 for every group member g: the value-norm GEMM over W_O's own slice
  VnormArgs v{};
  v.rq = pl.rq;
  v.src = kv_source(kv);
  v.v = static_cast<const uint16_t*>(kv->v);
  v.stride_req = kv->stride_req;
  v.stride_head = kv->stride_head;
  v.stride_tok = kv->stride_tok;
  v.D = pl.D;
  v.Dw = pl.D;
  v.units_total = pl.unit_base[pl.B];
  for (int b = 0; b <= pl.B; ++b) v.unit_base[b] = pl.unit_base[b];
  for (int b = 0; b < pl.B; ++b) v.blocks_per_head[b] = pl.blocks_per_head[b];
  v.grid_cap = pl.num_sms;
  v.wc = wait_ctl(pl, ws);
  for (int g = 0; g < pl.G; ++g) {
    float* nu_g = reinterpret_cast<float*>(wsb + L.nu) + static_cast<size_t>(g) * pl.n_scores;
    if ((rc = launch_rc(cudaMemsetAsync(nu_g, 0, static_cast<size_t>(pl.n_scores) * sizeof(float), st)))) return rc;
    CUtensorMap tw;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(pl.D),
                                static_cast<cuuint64_t>(pl.H)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(pl.H) * pl.G * kHeadDim * 2,
                                   static_cast<cuuint64_t>(pl.G) * kHeadDim * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(vnorm_w_tile_rows()), 1};
    if (!encode(&tw, static_cast<const uint16_t*>(w_o) + static_cast<size_t>(g) * kHeadDim, 3, dims, strides, box))
      return KVSEL_EINVAL;
    v.nu = nu_g;
    if ((rc = launch_rc(launch_vnorm(v, tw, st)))) return rc;
  }
  if ((rc = launch_rc(launch_perturb_stats(a, tq, tk, st)))) return rc;
  if ((rc = launch_rc(launch_perturb_accum(a, tq, tk, tv, st)))) return rc;
  return launch_rc(launch_perturb_finish(a, static_cast<const uint16_t*>(w_o), st));
}

int kvsel_run_anchors(const kvsel_params* p, const void* q, const kvsel_kv* kv, const float* rand_keys,
                      float* s_attn, int32_t* idx, int32_t* counts, int64_t* offsets, void* anchor_k, void* anchor_v,
                      int32_t* slot_k, float* gamma_k, int32_t* slot_v, float* gamma_v, void* ws, size_t ws_bytes,
                      void* stream) {
  Plan pl;
  int rc = make_plan(p, pl, true);
  if (rc) return rc;
  if (!q || !aligned16(q) || !s_attn || !rand_keys) return KVSEL_EINVAL;
  if (pl.qa && kv && kv->layout != KVSEL_LAYOUT_CONTIGUOUS) return KVSEL_EUNSUPPORTED;
  if ((rc = check_anchor_args(pl, kv, anchor_k, anchor_v, idx, counts, offsets, slot_k, gamma_k, slot_v, gamma_v, ws,
                              ws_bytes)))
    return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (pl.n_scores == 0) return KVSEL_OK;
  // pooling runs inside the selection kernel when the halo fits (as in kvsel_run_layer)
  const bool fuse_pool = (!p->pool || p->pool_kernel / 2 <= 32);
  if ((rc = do_score(p, pl, q, kv, nullptr, s_attn, nullptr, ws, st, !fuse_pool))) return rc;
  {
    StageScope sc(KVSEL_STAGE_SELECT, st);
    if (fuse_pool) {
      const float* raw = reinterpret_cast<const float*>(static_cast<uint8_t*>(ws) + pl.ws_sraw);
      rc = do_select(p, pl, s_attn, rand_keys, idx, counts, offsets, st, raw, nullptr, s_attn, nullptr);
    } else {
      rc = do_select(p, pl, s_attn, rand_keys, idx, counts, offsets, st);
    }
  }
  if (rc) return rc;
  if (pl.n_kept > 0 && (rc = do_compact(pl, kv, idx, counts, offsets, anchor_k, anchor_v, ws, st))) return rc;
  return do_anchor_project(pl, kv, anchor_k, anchor_v, idx, counts, offsets, slot_k, gamma_k, slot_v, gamma_v, ws, st);
}


uint64_t kvsel_launch_count(void) { return kvsel::g_launches.load(std::memory_order_relaxed); }

int kvsel_head_scores(const kvsel_params* p, const float* scores, float* head_out, void* stream) {
  Plan pl;
  const int rc = make_plan(p, pl, false);
  if (rc) return rc;
  if (!scores || !head_out) return KVSEL_EINVAL;
  if (pl.n_scores == 0 && pl.B * pl.H == 0) return KVSEL_OK;
  return launch_rc(launch_head_max(pl.rq, scores, head_out, static_cast<cudaStream_t>(stream)));
}

const char* kvsel_version(void) { return "kvsel 0.1 (sm_103a)"; }

const char* kvsel_strerror(int code) {
  switch (code) {
    case KVSEL_OK: return "ok";
    case KVSEL_EINVAL: return "invalid argument (pointer, alignment, size or enum)";
    case KVSEL_EBUDGET: return "budget below the forced entries or above the number of entries";
    case KVSEL_EUNSUPPORTED: return "unsupported configuration";
    case KVSEL_EWORKSPACE: return "workspace missing, misaligned or too small";
    case KVSEL_ECUDA: return "CUDA call or kernel launch failed";
    case KVSEL_ETIMEOUT: return "a bounded device-side wait ran out";
    case KVSEL_EDEVICE: return "device-side error (out-of-range index skipped)";
    default: return "unknown error";
  }
}

void kvsel_set_stage_events(void* const* events) { t_stage_events = events; }

int kvsel_workspace_size(const kvsel_params* p, size_t* bytes) {
  if (!bytes) return KVSEL_EINVAL;
  Plan pl;
  const int rc = make_plan(p, pl, true);
  if (rc) return rc;
  *bytes = pl.ws_total;
  return KVSEL_OK;
}

int kvsel_prepared_w_o_size(const kvsel_params* p, size_t* bytes) {
  if (!bytes) return KVSEL_EINVAL;
  Plan pl;
  const int rc = make_plan(p, pl, false);
  if (rc) return rc;
  if (!p->value_aware) return KVSEL_EINVAL;
  *bytes = pl.l2 ? static_cast<size_t>(pl.H) * 2 * kHeadDim * kHeadDim * 2
                 : static_cast<size_t>(pl.H) * pl.Dw * kHeadDim * 2;
  return KVSEL_OK;
}

int kvsel_prepare_w_o(const kvsel_params* p, const void* w_o, void* w_prep, size_t w_prep_bytes, void* ws,
                      size_t ws_bytes, void* stream) {
  if (!p) return KVSEL_EINVAL;
  kvsel_params q = *p;
  q.w_o_prepared = 0;   // the plan of the unprepared call: W_O in, its derived weights out
  Plan pl;
  int rc = make_plan(&q, pl, true);
  if (rc) return rc;
  if (!q.value_aware || !w_o || !aligned16(w_o) || !w_prep || (reinterpret_cast<uintptr_t>(w_prep) & 255u))
    return KVSEL_EINVAL;
  if (w_prep_bytes < pl.prep_bytes) return KVSEL_EINVAL;
  if (pl.l2 && (rc = check_ws(pl, ws, ws_bytes))) return rc;   // the L1 weights need no scratch
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (pl.l2) {
    CUtensorMap two;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(pl.H) * pl.G * kHeadDim, static_cast<cuuint64_t>(pl.D)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pl.H) * pl.G * kHeadDim * 2};
    const cuuint32_t box[2] = {64, 64};
    if (!encode(&two, w_o, 2, dims, strides, box)) return KVSEL_EINVAL;
    float* gpart = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.ws_gpart);
    return launch_rc(launch_value_gram(two, gpart, static_cast<uint16_t*>(w_prep), pl.H, pl.G, pl.D,
                                       wait_ctl(pl, ws), st));
  }
  return launch_rc(launch_wbar(static_cast<const uint16_t*>(w_o), static_cast<uint16_t*>(w_prep), pl.H, pl.G, pl.D,
                               q.wo_mode, nullptr, 0, st));
}

int kvsel_query_agnostic_split(const kvsel_params* p, int32_t* key_blocks, int32_t* row_splits) {
  if (!key_blocks || !row_splits) return KVSEL_EINVAL;
  Plan pl;
  const int rc = make_plan(p, pl, true);
  if (rc) return rc;
  if (!pl.qa) return KVSEL_EINVAL;
  *key_blocks = pl.qa_key_blocks;
  *row_splits = pl.qa_row_splits;
  return KVSEL_OK;
}

int kvsel_output_size(const kvsel_params* p, int64_t* n_scores, int64_t* n_kept, int64_t* n_segments) {
  Plan pl;
  const int rc = make_plan(p, pl, false);
  if (rc) return rc;
  if (n_scores) *n_scores = pl.n_scores;
  if (n_kept) *n_kept = pl.n_kept;
  if (n_segments) *n_segments = static_cast<int64_t>(pl.B) * pl.H;
  return KVSEL_OK;
}

int kvsel_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kStatusBytes) return KVSEL_EWORKSPACE;
  // status word and, when the workspace holds them, the grid-barrier counters (they reset
  // themselves after every use, so one zeroing at allocation is enough)
  const size_t n = ws_bytes >= kStatusBytes + kCounterBytes ? kStatusBytes + kCounterBytes : kStatusBytes;
  return launch_rc(cudaMemsetAsync(ws, 0, n, static_cast<cudaStream_t>(stream)));
}

int kvsel_score(const kvsel_params* p, const void* q, const kvsel_kv* kv, const void* w_o, float* s_attn,
                float* s_val, void* ws, size_t ws_bytes, void* stream) {
  Plan pl;
  int rc = make_plan(p, pl, true);
  if (rc) return rc;
  if (!q || !aligned16(q) || !s_attn) return KVSEL_EINVAL;
  if (p->value_aware && (!w_o || !aligned16(w_o) || !s_val)) return KVSEL_EINVAL;
  if ((rc = check_kv(kv, pl, p->value_aware != 0))) return rc;
  if (pl.qa && kv->layout != KVSEL_LAYOUT_CONTIGUOUS) return KVSEL_EUNSUPPORTED;
  if ((rc = check_ws(pl, ws, ws_bytes))) return rc;
  return do_score(p, pl, q, kv, w_o, s_attn, s_val, ws, static_cast<cudaStream_t>(stream));
}

int kvsel_select(const kvsel_params* p, const float* s_attn, const float* s_val, int32_t* idx, int32_t* counts,
                 int64_t* offsets, void* ws, size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  Plan pl;
  const int rc = make_plan(p, pl, false);
  if (rc) return rc;
  if (!s_attn || !idx || !counts || !offsets || ((p->value_aware || pl.anchor) && !s_val)) return KVSEL_EINVAL;
  if (pl.n_scores == 0) return KVSEL_OK;
  return do_select(p, pl, s_attn, s_val, idx, counts, offsets, static_cast<cudaStream_t>(stream));
}

int kvsel_compact(const kvsel_params* p, const kvsel_kv* kv, const int32_t* idx, const int32_t* counts,
                  const int64_t* offsets, void* k_out, void* v_out, void* ws, size_t ws_bytes, void* stream) {
  Plan pl;
  int rc = make_plan(p, pl, false);
  if (rc) return rc;
  if (!idx || !counts || !offsets || !k_out || !v_out || !aligned16(k_out) || !aligned16(v_out)) return KVSEL_EINVAL;
  if ((rc = check_kv(kv, pl, true))) return rc;
  if (ws && ws_bytes < kStatusBytes) return KVSEL_EWORKSPACE;
  if (pl.n_kept == 0) return KVSEL_OK;
  return do_compact(pl, kv, idx, counts, offsets, k_out, v_out, ws, static_cast<cudaStream_t>(stream));
}

int kvsel_partition(const kvsel_params* p, const kvsel_kv* kv, const int32_t* idx, const int32_t* counts,
                    const int64_t* offsets, int32_t* ev_idx, int32_t* ev_counts, int64_t* ev_offsets, void* k_ev,
                    void* v_ev, void* k_kept, void* v_kept, void* ws, size_t ws_bytes, void* stream) {
  Plan pl;
  int rc = make_plan(p, pl, false);
  if (rc) return rc;
  if (pl.anchor) return KVSEL_EUNSUPPORTED;
  const long long n_ev = pl.n_scores - pl.n_kept;
  if (!idx || !counts || !offsets || !ev_counts || !ev_offsets) return KVSEL_EINVAL;
  if (n_ev > 0 && (!ev_idx || !k_ev || !v_ev || !aligned16(k_ev) || !aligned16(v_ev))) return KVSEL_EINVAL;
  if ((k_kept == nullptr) != (v_kept == nullptr)) return KVSEL_EINVAL;
  if (k_kept && (!aligned16(k_kept) || !aligned16(v_kept))) return KVSEL_EINVAL;
  if ((rc = check_kv(kv, pl, true))) return rc;
  if (ws && ws_bytes < kStatusBytes) return KVSEL_EWORKSPACE;
  PartitionArgs a{};
  a.rq = pl.rq;
  a.src = kv_source(kv);
  a.k = static_cast<const uint16_t*>(kv->k);
  a.v = static_cast<const uint16_t*>(kv->v);
  a.stride_req = kv->stride_req;
  a.stride_head = kv->stride_head;
  a.stride_tok = kv->stride_tok;
  a.idx = idx;
  a.counts = counts;
  a.offsets = offsets;
  a.n_kept = pl.n_kept;
  a.n_evicted = n_ev;
  a.ev_idx = ev_idx;
  a.ev_counts = ev_counts;
  a.ev_offsets = ev_offsets;
  a.k_ev = static_cast<uint16_t*>(k_ev);
  a.v_ev = static_cast<uint16_t*>(v_ev);
  a.k_kept = static_cast<uint16_t*>(k_kept);
  a.v_kept = static_cast<uint16_t*>(v_kept);
  a.status = static_cast<int*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  StageScope sc(KVSEL_STAGE_COMPACT, st);
  return launch_rc(launch_partition(a, pl.n_max, st));
}

int kvsel_run_layer(const kvsel_params* p, const void* q, const kvsel_kv* kv, const void* w_o, float* s_attn,
                    float* s_val, int32_t* idx, int32_t* counts, int64_t* offsets, void* k_out, void* v_out, void* ws,
                    size_t ws_bytes, void* stream) {
  Plan pl;
  int rc = make_plan(p, pl, true);
  if (rc) return rc;
  if (pl.anchor) return KVSEL_EUNSUPPORTED;   // anchors: kvsel_run_anchors
  if (!q || !aligned16(q) || !s_attn || !idx || !counts || !offsets) return KVSEL_EINVAL;
  // no outputs for the rows: score and select only (the caller compacts later)
  const bool compact = k_out != nullptr || v_out != nullptr;
  if (compact && (!k_out || !v_out || !aligned16(k_out) || !aligned16(v_out))) return KVSEL_EINVAL;
  if (p->value_aware && (!w_o || !aligned16(w_o) || !s_val)) return KVSEL_EINVAL;
  if ((rc = check_kv(kv, pl, compact || p->value_aware))) return rc;
  if (pl.qa && kv->layout != KVSEL_LAYOUT_CONTIGUOUS) return KVSEL_EUNSUPPORTED;
  if ((rc = check_ws(pl, ws, ws_bytes))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (pl.n_scores == 0) return KVSEL_OK;
  // pooling and the value combination run inside the selection kernel when possible
  const bool fuse_pool = (!p->pool || p->pool_kernel / 2 <= 32);
  if ((rc = do_score(p, pl, q, kv, w_o, s_attn, s_val, ws, st, !fuse_pool))) return rc;
  if (fuse_pool) {
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    const float* raw = reinterpret_cast<const float*>(wsb + pl.ws_sraw);
    const float* nu = p->value_aware ? reinterpret_cast<const float*>(wsb + pl.ws_nu) : nullptr;
    if ((rc = do_select(p, pl, s_attn, s_val, idx, counts, offsets, st, raw, nu, s_attn,
                        p->value_aware ? s_val : nullptr)))
      return rc;
  } else if ((rc = do_select(p, pl, s_attn, s_val, idx, counts, offsets, st))) {
    return rc;
  }
  if (pl.n_kept == 0 || !compact) return KVSEL_OK;
  return do_compact(pl, kv, idx, counts, offsets, k_out, v_out, ws, st);
}

int kvsel_get_device_status(void* ws, void* stream, int* status) {
  if (!status) return KVSEL_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // no workspace: the built-in buffer of kvsel_score_noalloc on the current device
  if (!ws && noalloc_scratch_address(st, &ws) != KVSEL_OK) return KVSEL_ECUDA;
  int word = 0;
  if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return KVSEL_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KVSEL_ECUDA;
  if (word) {
    if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return KVSEL_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVSEL_ECUDA;
  }
  if (word & (DEV_TIMEOUT_PIPE | DEV_TIMEOUT_DRAIN))
    *status = KVSEL_ETIMEOUT;
  else if (word)
    *status = KVSEL_EDEVICE;
  else
    *status = KVSEL_OK;
  return KVSEL_OK;
}

}  // extern "C"
