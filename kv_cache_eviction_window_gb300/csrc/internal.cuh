// Internal declarations shared by the C-ABI host layer and the kernel translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace kvsel {

constexpr int kMaxBatch = 128;
constexpr int kHeadDim = 128;
// workspace layout: device status word, then the fused scoring kernel's grid-barrier
// counters (an arrival and a departure count per (request, head)), then the plan's buffers
constexpr size_t kStatusBytes = 256;
// counts every kernel launch (or graph capture of one) made by this library
void note_launch();

constexpr size_t kCounterBytes = 2 * 4 * static_cast<size_t>(kMaxBatch) * 64;

// Per-request table passed by value to kernels.
struct ReqTable {
  int B;                          // requests
  int H;                          // KV heads
  int n[kMaxBatch];               // context length of request b
  long long soff[kMaxBatch];      // offset of request b in the packed score arrays
};

// Where K/V tiles come from: a 4-D tensor map over the contiguous cache
// (d, token, head, request) or over the block pool (d, head, slot, block).
struct KvSource {
  int paged;
  int block_size;
  int max_blocks;
  int num_blocks;
  const int* block_table;   // device [B][max_blocks]
};

// TMA loads of `rows` tokens [tok0, tok0 + rows) of KV head h of request b into a
// K-major 128B-swizzled tile [2 column halves][rows][128 B].
__device__ __forceinline__ void load_kv_tile(const CUtensorMap* map, const KvSource& src, int b, int h, int n,
                                             int tok0, int rows, uint8_t* dst, uint64_t* bar, int* status) {
  const int half = rows * 128;
  if (!src.paged) {
    tma_load_4d(dst, map, bar, 0, tok0, h, b);
    tma_load_4d(dst + half, map, bar, 64, tok0, h, b);
  } else {
    const int bs = src.block_size;
    const int nblk_req = (n + bs - 1) / bs;
    for (int j = 0; j < rows / bs; ++j) {
      const int lb = tok0 / bs + j;
      int pb = -1;
      if (lb < nblk_req && lb < src.max_blocks) pb = __ldg(src.block_table + (size_t)b * src.max_blocks + lb);
      if (pb < 0 || pb >= src.num_blocks) {
        if (lb < nblk_req) atomicOr(status, DEV_BAD_INDEX);
        pb = 0;  // tokens past the request (masked by the epilogue) or a bad entry
      }
      tma_load_4d(dst + j * bs * 128, map, bar, 0, h, 0, pb);
      tma_load_4d(dst + half + j * bs * 128, map, bar, 64, h, 0, pb);
    }
  }
}

// Key-range decomposition shared by the two window-scoring passes: every (b, h) is cut
// into chunks of `chunk_len` keys; chunk ids run request-major, then head, then chunk.
struct ChunkTable {
  int chunk_len;                  // multiple of 256
  int total;                      // chunks over all requests and heads
  int base[kMaxBatch + 1];        // first chunk id of request b
  int per_head[kMaxBatch];        // chunks per head of request b
  int pbase[kMaxBatch + 1];       // first partial slot of request b (per head: per_head rounded up to 4)
};

// Row-statistics partials of (b, h): [2][R_pad][nch_pad] floats (max, sum), chunk index
// fastest so that a row's partials are contiguous.
__host__ __device__ inline int chunk_pad(int per_head) { return (per_head + 3) & ~3; }

struct WinScoreArgs {
  ReqTable rq;
  ChunkTable ck;
  KvSource src;
  int G, W, R, R_pad;             // R = G*W window rows per KV head, R_pad = roundup(R, 32)
  int causal;
  int reduce;                     // KVSEL_REDUCE_*
  float s2;                       // logit scale * log2(e)
  float* part;                    // per (b, h): [2][R_pad][chunk_pad]: row max (log2 units) and sum
  float* s_raw;                   // packed [sum_b H*n_b] reduced scores
  float* nu_zero;                 // optional, packed like s_raw: zeroed by the fused launch for
                                  // the value-norm kernel that accumulates into it next
  WaitCtl wc;
};

// Query-agnostic scoring (all G*n query rows of a KV head, non-causal, max reduction).
struct QaArgs {
  int H;                          // KV heads
  int n;                          // keys (context length)
  int GN;                         // query rows per head (G * n)
  int row_blocks;                 // pass 1: blocks of 512 query rows per head
  int key_blocks;                 // pass 2: blocks of 256 keys per head
  int row_splits;                 // pass 2: query-row slices per key block
  float s2;                       // logit scale * log2(e)
  float* c2;                      // [H][GN] row log-sum-exp, log2 units
  uint32_t* tmax;                 // [H][n] order-preserving keys of max_r (l*s2 - c2_r)
  float* s_raw;                   // [H][n] exp2 of that max (softmax), or the max logit itself
  int logit;                      // softmax-free score: no row log-sum-exp, s2 = scale, c2 = 0
  WaitCtl wc;
};
cudaError_t launch_qa_rowlse(const QaArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t st);
cudaError_t launch_qa_keymax(const QaArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t st);
int qa_block_rows();    // pass 1: query rows per CTA
int qa_key_block();     // pass 2: keys per CTA
int qa_query_tile();    // pass 2: query rows per streamed tile

struct VnormArgs {
  ReqTable rq;
  KvSource src;
  const uint16_t* v;              // value cache (contiguous) or value block pool (paged)
  long long stride_req, stride_head, stride_tok;   // contiguous layout, in elements
  int D;                          // rows of W_O (output features)
  int Dw;                         // rows of the combined weight per head (D or G*D)
  int units_total;                // (b, h, token block) work units
  int unit_base[kMaxBatch + 1];   // first unit of request b
  int blocks_per_head[kMaxBatch]; // token blocks per head of request b
  float* nu;                      // packed [sum_b H*n_b]
  int grid_cap;                   // CTAs at most (the call's SM budget); 0 = every SM
  WaitCtl wc;
};

// L2 value norm through the Gram matrix Gamma_h = W_h^T W_h.  Units are (request, head,
// 128-token block), request-major then head, as VnormArgs with 128-token blocks.
struct VgramArgs {
  ReqTable rq;
  KvSource src;
  int units_total;
  int unit_base[kMaxBatch + 1];
  int blocks_per_head[kMaxBatch];
  float* nu;                      // packed [sum_b H*n_b]
  int grid_cap;                   // CTAs at most (the call's SM budget); 0 = every SM
  WaitCtl wc;
};
// Row slices of the Gram partials (workspace: H * slices * 128 * 128 fp32).
int gram_slices(int Dw);
// Gamma partials (part) straight from W_O, then Gamma hi/lo (gam: [H][2][d][d] bf16).
// two: 2-D map over W_O (H*G*d columns, D rows), box 64 x 64, 128-byte swizzle.  G <= 8.
cudaError_t launch_value_gram(const CUtensorMap& two, float* part, uint16_t* gam, int H, int G, int D, WaitCtl wc,
                              cudaStream_t st);
// tv: V tiles of 128 tokens (kv_map); tg: 2-D map over gam (d, H*2*d rows), box 64 x 128.
cudaError_t launch_vgram(const VgramArgs& a, const CUtensorMap& tv, const CUtensorMap& tg, cudaStream_t st);

// AnchorKV nearest-anchor projection.  Units are (request, head, side, 128-token tile):
// request-major, then head, then side (K = 0, V = 1), then tile.
struct AnchorArgs {
  ReqTable rq;
  KvSource src;
  int units_total;
  int unit_base[kMaxBatch + 1];
  int tiles[kMaxBatch];            // 128-token tiles per head of request b
  const int32_t* idx;              // anchor positions, ascending within each segment
  const int32_t* counts;           // anchors per segment (b, h)
  const int64_t* offsets;          // first anchor row of each segment
  long long n_rows;                // rows of the compacted anchor buffers
  const float* inv;                // [2][n_rows]: 1 / |a| of the K and V anchor rows
  int32_t* slot[2];                // K, V: anchor slot per position (packed like scores)
  float* gamma[2];                 // K, V: projection coefficient per position
  WaitCtl wc;
};
int anchor_max();
cudaError_t launch_anchor_norms(const uint16_t* ak, const uint16_t* av, long long rows, float* inv, cudaStream_t st);
cudaError_t launch_anchor_project(const AnchorArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const CUtensorMap& tak, const CUtensorMap& tav, cudaStream_t st);

// Output perturbation of a kept set (CriticalKV Theorems 3.2, 3.3, C.1) for the window rows
// of every KV head.  Key chunks as in ChunkTable; rows r = g * W + w (R = G * W <= 128).
struct PerturbArgs {
  ReqTable rq;
  ChunkTable ck;
  KvSource src;
  int G, W, R;
  int causal;
  float s2;                       // logit scale * log2(e)
  int D;                          // rows of W_O
  const uint8_t* keep;            // packed [sum_b H*n_b]: 1 = kept
  const float* nu;                // [G][n_scores]: ||W_O^(h,g) v_i||_1 per query head of the group
  long long n_scores;
  float* stat_part;               // [chunks][128][7]: m (log2), Z, Z_S, Z_N, C_N, P_S, max partials
  float* stat;                    // [B*H][128][7] merged
  float* e_part;                  // [chunks][128][128]: sum_i c_ri v_i partials
  float* e;                       // [B*H][128][128] merged
  float* y_part;                  // [B*H*G][D/256][W]: partial ||W_O^(h,g) e_r||_1
  float* out;                     // [B][H][3][G][W]: actual, bound, relaxed bound
  WaitCtl wc;
};
cudaError_t launch_perturb_mask(const ReqTable& rq, const int32_t* idx, const int32_t* counts, const int64_t* offsets,
                                int max_count, uint8_t* keep, int* status, cudaStream_t st);
cudaError_t launch_perturb_stats(const PerturbArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t st);
cudaError_t launch_perturb_accum(const PerturbArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, cudaStream_t st);
cudaError_t launch_perturb_finish(const PerturbArgs& a, const uint16_t* w_o, cudaStream_t st);
int perturb_slices(int D);   // 256-feature slices of W_O rows in the projection

// Device address of kvsel_score_noalloc's built-in scratch buffer in the current context
// (KVSEL_OK, or KVSEL_ECUDA when it cannot be looked up).
int noalloc_scratch_address(cudaStream_t st, void** out);

// Raise a kernel's dynamic shared-memory limit once per device (cached).
cudaError_t ensure_smem(const void* func, size_t bytes);

// Host-side launchers (return cudaError_t of the launch).
cudaError_t launch_win_rowstats(const WinScoreArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, int mt,
                                cudaStream_t st);
cudaError_t launch_win_keysum(const WinScoreArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t st);
cudaError_t launch_win_fused(const WinScoreArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                             unsigned int* grid_count, cudaStream_t st);


// Also zeroes nu[0, nu_count), which launch_vnorm (next on the stream) accumulates into.
cudaError_t launch_wbar(const uint16_t* w_o, uint16_t* wbar, int H, int G, int D, int wo_mode, float* nu,
                        long long nu_count, cudaStream_t st);
cudaError_t launch_vnorm(const VnormArgs& a, const CUtensorMap& tw, cudaStream_t st);
int vnorm_token_block();
int vnorm_w_tile_rows();

// Per-segment maximum of a packed score array: out[b*H + h] = max_i s[soff[b] + h*n_b + i]
// (-inf for an empty request).
cudaError_t launch_head_max(const ReqTable& rq, const float* s, float* out, cudaStream_t st);

cudaError_t launch_finalize(const ReqTable& rq, const float* s_raw, const float* nu, float* s_attn, float* s_val,
                            int pool, int pool_kernel, float eps, cudaStream_t st);

// Selection.  One cluster of CTAs per segment (b, h) in per-head mode, per request in
// per-layer mode.
struct SelectArgs {
  ReqTable rq;
  int mode;                       // KVSEL_BUDGET_*
  int two_stage;
  float alpha;
  int n_sink, n_recent;
  int budget[kMaxBatch];          // per head (per-head mode) or per layer (per-layer mode)
  int budget1[kMaxBatch];         // two-stage: stage-1 budget max(floor(alpha*B), |F|)
  int floor_h[kMaxBatch];         // per-layer mode: per-head floor
  const float* s1;                // stage-1 scores (s_attn)
  const float* s2;                // stage-2 scores (s_val) or null
  // pooling fused into the selection (kvsel_run_layer): when raw != null the kernel pools
  // raw (and combines with nu), writes out_attn / out_val, and selects on those values
  const float* raw;
  const float* nu;
  float* out_attn;
  float* out_val;
  int pool, pool_kernel;
  float eps;
  int32_t* idx;
  int32_t* counts;
  int64_t* offsets;               // written for every segment
  long long seg_out[kMaxBatch];   // output offset of request b's first segment
  // per-head mode with budgets set on the device (value-aware selection under a per-layer
  // budget): segment s keeps dev_counts[s] entries at dev_offsets[s]; counts and offsets
  // are then not rewritten
  const int32_t* dev_counts;
  const int64_t* dev_offsets;
};
cudaError_t launch_select(const SelectArgs& a, int cluster, int chunk_cap, cudaStream_t st);
// min_cs: 0 for a call alone on the device, else the smallest cluster to try (calls overlap)
int select_cluster_size(int max_len, int segments, int min_cs, int* chunk_cap);

struct CompactArgs {
  ReqTable rq;
  KvSource src;
  const uint16_t* k;
  const uint16_t* v;
  long long stride_req, stride_head, stride_tok;
  const int32_t* idx;
  const int32_t* counts;
  const int64_t* offsets;
  uint16_t* k_out;
  uint16_t* v_out;
  long long n_kept;               // rows of k_out / v_out
  int* status;                    // may be null
};
cudaError_t launch_compact(const CompactArgs& a, int max_count, int num_sms, cudaStream_t st);

// Partition of every segment into kept and evicted positions with both sides' rows
// (kvsel_partition).  Grid: (64-position tiles of the longest request, segments).
struct PartitionArgs {
  ReqTable rq;
  KvSource src;
  const uint16_t* k;
  const uint16_t* v;
  long long stride_req, stride_head, stride_tok;
  const int32_t* idx;             // kept positions, ascending per segment
  const int32_t* counts;
  const int64_t* offsets;
  long long n_kept;               // rows of idx / k_kept / v_kept
  long long n_evicted;            // rows of ev_idx / k_ev / v_ev
  int32_t* ev_idx;                // evicted positions, ascending per segment
  int32_t* ev_counts;
  int64_t* ev_offsets;
  uint16_t* k_ev;
  uint16_t* v_ev;
  uint16_t* k_kept;               // may be null (then v_kept is null too)
  uint16_t* v_kept;
  int* status;                    // may be null
};
cudaError_t launch_partition(const PartitionArgs& a, int n_max, cudaStream_t st);


}  // namespace kvsel
