/*
 * kvsel.h — end-of-prefill KV-cache importance scoring, top-B selection and compaction
 * on one NVIDIA GB300 (sm_103a).
 *
 * The operations follow the pages this library restates:
 *   - Observation-window scoring: the last W prompt queries of each GQA group attend to
 *     all n cached keys; the fp32 softmax weights are reduced over window rows and the
 *     G query heads of the group, then 1-D pooled along the sequence
 *     ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", §3.4 Algorithm 2;
 *     SnapKV kernel 7 / window 32 per its §4.1).
 *   - Value-aware criterion (A + eps) * ||W_O v||_1 and two-stage selection with
 *     alpha = 0.5 (same page, §3.3 Theorem 3.3, §3.4 Algorithm 1, §3.5, footnote 3).
 *   - Query-agnostic maximum cross-attention score, its softmax-free variant
 *     (KVzip-logit) and head-level scores, and a budget shared by the heads of a layer
 *     ("KVzip: Query-Agnostic KV Cache Compression with Context Reconstruction", §3.2,
 *     §3.4, §3.6, §4.2, §6.5).
 *   - Attention sinks and the recent window are always kept ("VestigeKV: The NoPE-MLA KV
 *     Cache Carries Its Own Eviction Signal in a Vestigial Branch", §4.1; "AnchorKV:
 *     Anchor-Residual KV Cache Compression", §3.2).
 *   - Eviction acts on the un-replicated KV heads; the result is a per-head
 *     variable-length cache (KVzip §4.2, §7.1).
 *
 * Conventions (all entry points):
 *   - Every pointer named device is a CUDA device pointer, 16-byte aligned; bf16 data is
 *     IEEE bfloat16.  Host pointers are marked host.
 *   - The caller owns every buffer.  The library never allocates device or host memory;
 *     scratch space is the caller's workspace (kvsel_workspace_size).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are asynchronous
 *     on that stream; argument errors are returned before anything is launched.
 *   - Return value: KVSEL_OK or a negative KVSEL_E* code (kvsel_strerror).  Errors found
 *     on the device (a bounded wait that ran out) are recorded in the workspace's status
 *     word and read with kvsel_get_device_status after the stream work.
 *   - head_dim must be 128.
 *
 * Data layouts (row-major, innermost last):
 *   q (window scoring)         [batch][h_kv][group][window][head_dim] bf16
 *   q (query-agnostic, window=0) [h_kv][group][n_ctx][head_dim]      bf16, batch 1
 *   k, v (contiguous)          element (b, h, i, c) at b*stride_req + h*stride_head
 *                              + i*stride_tok + c (elements; stride_tok >= head_dim)
 *   k, v (paged)               pool [num_blocks][block_size][h_kv][head_dim]; token i of
 *                              request b is slot i % block_size of block
 *                              block_table[b*max_blocks + i / block_size]
 *   w_o                        [d_model][h_kv*group*head_dim] bf16 (nn.Linear weight);
 *                              query head h*group+g owns columns [(h*group+g)*d, +d)
 *   scores (s_attn, s_val)     fp32, packed by request: request b starts at
 *                              h_kv * (n_0 + ... + n_{b-1}); head h of it at + h*n_b
 *   idx                        int32 token positions, ascending within each (b, h)
 *                              segment; segment (b, h) starts at offsets[b*h_kv + h]
 *   counts / offsets           [batch*h_kv] int32 / int64 (exclusive prefix sum of counts)
 *   k_out, v_out               [total kept][head_dim] bf16, same packing as idx
 */
#ifndef KVSEL_H
#define KVSEL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------ */
#define KVSEL_OK 0
#define KVSEL_EINVAL (-1)        /* NULL / misaligned pointer, bad size or enum value    */
#define KVSEL_EBUDGET (-2)       /* forced entries exceed the budget, or budget > n*H    */
#define KVSEL_EUNSUPPORTED (-3)  /* valid request outside what the kernels implement    */
#define KVSEL_EWORKSPACE (-4)    /* workspace NULL or smaller than kvsel_workspace_size  */
#define KVSEL_ECUDA (-5)         /* a CUDA runtime/driver call or launch failed          */
#define KVSEL_ETIMEOUT (-6)      /* a bounded device-side wait ran out (status word)     */
#define KVSEL_EDEVICE (-7)       /* other device-side error recorded in the status word  */

/* ---- enumerations ------------------------------------------------------------------- */
/* MAX_LOGIT: query-agnostic only — the maximum scaled dot product itself, without
 * softmax normalisation (KVzip §6.5, "KVzip-logit"). */
enum { KVSEL_REDUCE_SUM = 0, KVSEL_REDUCE_MEAN = 1, KVSEL_REDUCE_MAX = 2, KVSEL_REDUCE_MAX_LOGIT = 3 };
enum { KVSEL_POOL_NONE = 0, KVSEL_POOL_MAX = 1, KVSEL_POOL_AVG = 2 };
/* ANCHOR: AnchorKV anchors ("AnchorKV: Anchor-Residual KV Cache Compression", §3.2,
 * §4.1).  Per head k = floor(budget_ratio * n) anchors (1/128 on the page), at least the
 * forced entries and at most n; the forced entries (the recent window) count inside k;
 * floor(alpha * (k - |F|)) more go to the highest s_attn (alpha = rho = 0.7), the rest to
 * the largest of the caller's random keys, which kvsel_select takes in place of s_val:
 * i.i.d. uniform keys make that share a uniform draw without replacement.  Not with
 * value_aware; kvsel_run_layer refuses it (use kvsel_run_anchors). */
enum { KVSEL_BUDGET_PER_HEAD = 0, KVSEL_BUDGET_PER_LAYER = 1, KVSEL_BUDGET_ANCHOR = 2 };
enum { KVSEL_WO_GROUP_SUM = 0, KVSEL_WO_PER_HEAD = 1 };
/* Value norm of the value-aware criterion: L1 (CriticalKV's choice) or L2, the other
 * distance its App. C.3 compares.  L2 is computed through the d x d Gram matrix
 * W_h^T W_h (32x fewer flops at D = 4096); group-sum W_O reading only. */
enum { KVSEL_NORM_L1 = 0, KVSEL_NORM_L2 = 1 };
enum { KVSEL_LAYOUT_CONTIGUOUS = 0, KVSEL_LAYOUT_PAGED = 1 };

#define KVSEL_MAX_BATCH 128

/* ---- parameters --------------------------------------------------------------------- */
typedef struct kvsel_params {
  int32_t h_kv;         /* KV heads H                                                    */
  int32_t group;        /* query heads per KV head G (GQA, KVzip §2.2)                   */
  int32_t head_dim;     /* d; must be 128                                                */
  int32_t d_model;      /* D, rows of W_O (value-aware only); multiple of 128            */
  int32_t n_ctx;        /* context length n (all requests when n_ctx_per_req is NULL)    */
  int32_t window;       /* W observation-window queries per group head (Algorithm 2's
                           n'); 0 = query-agnostic scoring over all n positions (KVzip)  */
  int32_t q_chunk;      /* query-agnostic: query positions per chunk (KVzip §3.4); 0=all */
  int32_t causal;       /* 1: window row w (position n-W+w) sees keys <= n-W+w           */
  float scale;          /* logit scale; 0 = 1/sqrt(head_dim)                             */
  int32_t reduce;       /* KVSEL_REDUCE_*: over window rows and group heads              */
  int32_t pool;         /* KVSEL_POOL_*: 1-D pooling along n, stride 1, centred window   */
  int32_t pool_kernel;  /* odd pooling width k (max ignores out-of-range positions, avg
                           pads with zeros and divides by k)                             */
  int32_t value_aware;  /* 1: s_val = (s_attn + eps) * ||W_O v||_1 and two-stage select */
  int32_t wo_mode;      /* KVSEL_WO_*: GQA reading of W_O^h (group sum, default)         */
  float eps;            /* 1e-4 (CriticalKV footnote 3)                                  */
  float alpha;          /* first-stage share of the budget (0.5, CriticalKV §3.5)        */
  int32_t n_sink;       /* first n_sink positions always kept (4)                        */
  int32_t n_recent;     /* last n_recent positions always kept (W)                       */
  int32_t budget_mode;  /* KVSEL_BUDGET_*                                                */
  double budget_ratio;  /* per head: B = floor(ratio*n); per layer: floor(ratio*n*H)     */
  double floor_ratio;   /* per layer: each head keeps at least floor(floor_ratio*n)      */
  int32_t batch;        /* requests in the call (<= KVSEL_MAX_BATCH)                      */
  const int32_t* n_ctx_per_req; /* host [batch] context lengths, or NULL                  */
  int32_t value_norm;   /* KVSEL_NORM_*: ||W_h v||_1 (default) or ||W_h v||_2            */
  int32_t w_o_prepared; /* 1: the w_o argument of the scoring calls is the output of
                           kvsel_prepare_w_o for these parameters, not W_O itself        */
  uint64_t wait_cycles; /* bound of one device-side wait, in SM clock cycles; 0 = default
                           (2e9, about 1 s at the boost clock).  A wait that runs out ends
                           its kernel with KVSEL_ETIMEOUT in the device status word; 1
                           makes every wait that is not already satisfied give up at once */
  int32_t sm_budget;    /* SMs the call sizes its one-CTA-per-SM kernels for (the key
                           chunks of the scoring pass, the value-norm GEMM): 0 = every
                           SM of the device.  A smaller budget leaves SMs to calls
                           running at the same time on other streams (independent
                           layers), so that, e.g., two layers' scoring kernels run side
                           by side; the results do not depend on it beyond fp32 rounding
                           order                                                         */
  int32_t concurrent;   /* 1: other work may run on the device at the same time (calls
                           on other streams).  The call then uses only kernels that make
                           progress whatever else is resident: the two scoring passes run
                           as two launches.  0: when R <= 256 they run as one cooperative
                           launch whose CTAs wait for each other at a per-head barrier,
                           which needs every key chunk's CTA resident at once; two such
                           calls running at the same time can each hold SMs the other
                           waits for, until their bounded waits end them with
                           KVSEL_ETIMEOUT.  Set 1 whenever calls overlap.  With 1 the
                           selection also runs on clusters of 4 CTAs per segment instead of
                           8 or 16 (longer alone, half the SM time beside other calls), or
                           of 2 when 4 per segment would exceed sm_budget; results are the
                           same either way                                                */
} kvsel_params;

/* K/V cache view, contiguous or paged (block_size tokens per block). */
typedef struct kvsel_kv {
  const void* k;                /* device bf16                                          */
  const void* v;                /* device bf16                                          */
  int32_t layout;               /* KVSEL_LAYOUT_*                                       */
  int64_t stride_req;           /* contiguous: elements between requests                */
  int64_t stride_head;          /* contiguous: elements between heads                   */
  int64_t stride_tok;           /* contiguous: elements between tokens                  */
  const int32_t* block_table;   /* paged: device [batch][max_blocks]                    */
  int32_t block_size;           /* paged: tokens per block: 8, 16, 32 or 64             */
  int32_t max_blocks;           /* paged: row length of block_table                     */
  int32_t num_blocks;           /* paged: blocks in the pool                            */
} kvsel_kv;

/* ---- sizes --------------------------------------------------------------------------- */

/* Bytes of device workspace that kvsel_score / kvsel_select / kvsel_run_layer need for
 * these parameters on the current device.  Host-only; no CUDA work. */
int kvsel_workspace_size(const kvsel_params* p, size_t* bytes);

/* Output sizes: *n_scores = elements of s_attn / s_val (H * sum of n_b), *n_kept = total
 * kept entries (length of idx and rows of k_out / v_out), *n_segments = batch * h_kv
 * (length of counts / offsets).  Any output pointer may be NULL. */
int kvsel_output_size(const kvsel_params* p, int64_t* n_scores, int64_t* n_kept, int64_t* n_segments);

/* Zero the workspace's device status word (do once after allocating a workspace). */
int kvsel_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* ---- weights prepared once per model ------------------------------------------------------ */

/* Bytes of the prepared value-norm weights of kvsel_prepare_w_o (value_aware only):
 * L1 norm: W_h for every KV head, [h_kv][d_model][head_dim] bf16 (the per-head W_O reading:
 * [h_kv][group*d_model][head_dim]); L2 norm: Gamma_h = W_h^T W_h as a bf16 high part and
 * remainder, [h_kv][2][head_dim][head_dim].  Host-only. */
int kvsel_prepared_w_o_size(const kvsel_params* p, size_t* bytes);

/* The value-aware criterion projects each value through W_h, the sum of the group's W_O
 * column slices ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", §3.4 Algorithm 1, App.
 * D.4).  W_h depends on the model's weights alone, so it can be built once per model (per
 * layer) instead of inside every scoring call: this call writes it (or, for the L2 norm,
 * its Gram matrix) into w_prep; scoring calls whose params set w_o_prepared = 1 then take
 * w_prep as their w_o argument.  Results are bit-identical to passing W_O itself.
 *   w_o     device bf16 [d_model][h_kv*group*head_dim]
 *   w_prep  device, 256-byte aligned, kvsel_prepared_w_o_size bytes
 *   ws      L2 norm: device workspace of kvsel_workspace_size bytes (for params with
 *           w_o_prepared = 0; it holds the Gram partials); L1 norm: not used, may be NULL
 * Asynchronous on `stream`. */
int kvsel_prepare_w_o(const kvsel_params* p, const void* w_o, void* w_prep, size_t w_prep_bytes, void* ws,
                      size_t ws_bytes, void* stream);

/* ---- the path ------------------------------------------------------------------------ */

/* Score every cached key (CriticalKV Algorithm 2; KVzip §3.2 when window == 0).
 *   q       device bf16, layout above
 *   kv      K/V view (V is read only when value_aware)
 *   w_o     device bf16 [d_model][h_kv*group*head_dim], or NULL unless value_aware
 *   s_attn  device fp32 [n_scores]: pooled attention score
 *   s_val   device fp32 [n_scores]: (s_attn + eps) * nu, or NULL unless value_aware
 *           (nu = ||W_h v||_1, or ||W_h v||_2 with value_norm = KVSEL_NORM_L2)
 *   ws      device workspace of ws_bytes >= kvsel_workspace_size
 * Query-agnostic scoring (window == 0) supports batch 1, non-causal, reduce MAX (maximum
 * softmax weight) or MAX_LOGIT (maximum logit, no softmax: one pass instead of two). */
int kvsel_score(const kvsel_params* p, const void* q, const kvsel_kv* kv, const void* w_o, float* s_attn,
                float* s_val, void* ws, size_t ws_bytes, void* stream);

/* Select the kept entries from the scores (CriticalKV Algorithm 1 when value_aware;
 * per-layer budget with per-head floors, KVzip §4.2, when budget_mode is PER_LAYER).
 * Both together follow CriticalKV Algorithm 2: the layer budget is split over the heads
 * by the layer-wide top of s_attn (line 1, with the floors), then each head keeps its
 * share by the two-stage criterion (line 8).
 * Forced entries (sinks, recent window) are always kept and count inside the budget.
 *   s_attn  device fp32 [n_scores]; s_val device fp32 [n_scores] or NULL
 *   idx     device int32 [n_kept]; counts device int32 [batch*h_kv];
 *   offsets device int64 [batch*h_kv]
 * Order: score descending, ties by index ascending (flat index h*n+i per layer). */
int kvsel_select(const kvsel_params* p, const float* s_attn, const float* s_val, int32_t* idx, int32_t* counts,
                 int64_t* offsets, void* ws, size_t ws_bytes, void* stream);

/* Gather the kept K/V rows into dense per-segment buffers (bit-exact copies).
 *   idx/counts/offsets as produced by kvsel_select (device)
 *   k_out, v_out  device bf16 [n_kept][head_dim]
 * Indices outside [0, n_b) are flagged in the status word when ws != NULL; their output
 * rows are written as zeros.  k_out and v_out must be 16-byte aligned. */
int kvsel_compact(const kvsel_params* p, const kvsel_kv* kv, const int32_t* idx, const int32_t* counts,
                  const int64_t* offsets, void* k_out, void* v_out, void* ws, size_t ws_bytes, void* stream);

/* Partition every (request, KV head) segment into the kept positions and their complement,
 * the evicted ones, and write the rows of both sides ("VestigeKV: The NoPE-MLA KV Cache
 * Carries Its Own Eviction Signal in a Vestigial Branch", §4.1: eviction deletes nothing;
 * the evicted rows go to an archive, bit-exact, and every position lands in exactly one
 * of the two sides).  One pass reads every K/V row once and writes it once.
 *   idx/counts/offsets  device, the kept set as kvsel_select writes it (ascending per
 *            segment; offsets the exclusive prefix sum of counts from 0)
 *   ev_idx   device int32 [n_scores - n_kept]: evicted positions, ascending per segment
 *   ev_counts / ev_offsets  device int32 / int64 [batch*h_kv]: n_b - counts, and the
 *            exclusive prefix sum of ev_counts (segments in the same order as counts)
 *   k_ev, v_ev          device bf16 [n_scores - n_kept][head_dim]: the evicted rows, packed
 *            like ev_idx
 *   k_kept, v_kept      device bf16 [n_kept][head_dim] or both NULL: the kept rows, packed
 *            like idx (what kvsel_compact writes)
 *   ws       NULL, or a workspace of at least 256 bytes whose status word records entries
 *            found out of range (KVSEL_EDEVICE through kvsel_get_device_status)
 * A segment whose count or offset does not fit the buffers, or a kept list that is not
 * strictly ascending, is skipped (its rows are not written) and flagged in the status
 * word; nothing outside the buffers is touched.  Sizes: kvsel_output_size
 * (n_scores - n_kept evicted rows in all). */
int kvsel_partition(const kvsel_params* p, const kvsel_kv* kv, const int32_t* idx, const int32_t* counts,
                    const int64_t* offsets, int32_t* ev_idx, int32_t* ev_counts, int64_t* ev_offsets, void* k_ev,
                    void* v_ev, void* k_kept, void* v_kept, void* ws, size_t ws_bytes, void* stream);

/* score -> select -> compact for one layer, enqueued back to back on `stream`.
 * s_attn / s_val are written as in kvsel_score (s_val may be NULL when !value_aware).
 * k_out and v_out may both be NULL: the call then ends after the selection, for a
 * caller that gathers the kept rows itself later (kvsel_compact or kvsel_partition, for
 * example on another stream while the next layer is scored). */
int kvsel_run_layer(const kvsel_params* p, const void* q, const kvsel_kv* kv, const void* w_o, float* s_attn,
                    float* s_val, int32_t* idx, int32_t* counts, int64_t* offsets, void* k_out, void* v_out,
                    void* ws, size_t ws_bytes, void* stream);

/* ---- scoring without a caller-provided workspace --------------------------------------- */

/* Size of the library's built-in scratch buffer used by kvsel_score_noalloc (16 MiB:
 * enough for one layer of the 32K Llama-3.1-8B or 128K Qwen2.5-7B shapes). */
#define KVSEL_NOALLOC_SCRATCH_BYTES (16u << 20)

/* kvsel_score for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call: it exists for processes whose device memory belongs to an
 * arena or caching allocator (a serving engine that reserved its KV-cache pool up front)
 * and for code that must not call cudaMalloc/cudaFree because they can synchronise the
 * device.  Same arguments and results as kvsel_score minus the workspace: the scratch is
 * a fixed KVSEL_NOALLOC_SCRATCH_BYTES buffer inside the library, held on every GPU that
 * loads the library until the process exits.  No allocation of any kind is made.
 *   Returns KVSEL_EWORKSPACE when the request needs more scratch than that buffer
 *   (kvsel_workspace_size > KVSEL_NOALLOC_SCRATCH_BYTES), before any launch.
 *   All calls share the buffer, which keeps the last call's contents (each call zeroes the
 *   status word at its start, so read the status after a call and before the next one): calls whose GPU work overlaps race; serialise
 *   them.  The buffer's device address is looked up (cudaGetSymbolAddress) by every call
 *   made outside stream capture, in the calling thread's current context, and recorded
 *   for that context; a call under stream capture uses the recorded address, so make at
 *   least one call per context (device) before capturing any.  Errors found on the device
 *   (a bounded wait that ran out, a block-table entry out of range) are read and cleared
 *   with kvsel_get_device_status(NULL, stream, &status) on the same device. */
int kvsel_score_noalloc(const kvsel_params* p, const void* q, const kvsel_kv* kv, const void* w_o, float* s_attn,
                        float* s_val, void* stream);

/* ---- diagnostics --------------------------------------------------------------------- */

/* Synchronise `stream`, read and clear the workspace's device status word.  *status is
 * KVSEL_OK, KVSEL_ETIMEOUT (a bounded device wait ran out) or KVSEL_EDEVICE (an index or
 * block-table entry out of range was skipped).  ws == NULL reads and clears the status
 * word of the built-in buffer that kvsel_score_noalloc uses on the current device. */
int kvsel_get_device_status(void* ws, void* stream, int* status);

/* Stages of the path, in launch order within one layer. */
enum {
  KVSEL_STAGE_ROWSTATS = 0,  /* scoring pass 1 (row softmax statistics), or both    
                                passes when they run as one cooperative launch        */
  KVSEL_STAGE_KEYSUM = 1,    /* window scoring pass 2: per-key reduced probabilities */
  KVSEL_STAGE_WBAR = 2,      /* value-aware: W_O slices of each KV head, bf16        */
  KVSEL_STAGE_VNORM = 3,     /* value-aware: ||W_h v||_1 per token (tensor cores)    */
  KVSEL_STAGE_FINALIZE = 4,  /* pooling and (s + eps) * nu (inside the selection     
                                launch on the kvsel_run_layer path)                   */
  KVSEL_STAGE_SELECT = 5,    /* top-B selection                                      */
  KVSEL_STAGE_COMPACT = 6,   /* gather of the kept K/V rows                          */
  KVSEL_STAGE_PROJECT = 7,   /* anchors: anchor norms and nearest-anchor projection  */
  KVSEL_STAGE_PERTURB = 8,   /* output perturbation of a kept set (all its kernels)  */
  KVSEL_STAGE_COUNT = 9
};

/* Diagnostics: while `events` is non-NULL, each kernel launched by this thread's
 * subsequent calls is bracketed by cudaEventRecord(events[2*stage]) and
 * cudaEventRecord(events[2*stage + 1]) on the launch stream (NULL entries skipped).
 * `events` is a host array of 2*KVSEL_STAGE_COUNT cudaEvent_t created by the caller and
 * must stay valid until the hook is cleared with NULL.  No effect on results. */
void kvsel_set_stage_events(void* const* events);

/* Number of kernels this library has launched in this process so far (all devices and
 * threads; a launch recorded into a CUDA graph under stream capture counts once, at
 * capture).  The difference across a call is that call's kernel count.  Never fails. */
uint64_t kvsel_launch_count(void);

/* Diagnostics: how query-agnostic scoring (window == 0) splits its work on the current
 * device: *key_blocks = blocks of 256 keys per head, *row_splits = slices of the G*n query
 * rows per key block (the per-key maximum of each slice is merged with an atomic max).
 * Host-only; errors as kvsel_workspace_size, KVSEL_EINVAL when window != 0. */
int kvsel_query_agnostic_split(const kvsel_params* p, int32_t* key_blocks, int32_t* row_splits);

/* Head-level scores (KVzip §3.4, §3.6): head_out[b*h_kv + h] = the maximum over the
 * sequence of request b, head h of `scores` (packed as kvsel_score writes them, device fp32
 * [n_scores]); -inf for an empty request.  head_out: device fp32 [batch*h_kv].  Asynchronous
 * on `stream`; errors as kvsel_output_size. */
int kvsel_head_scores(const kvsel_params* p, const float* scores, float* head_out, void* stream);

/* ---- AnchorKV anchors ---------------------------------------------------------------- */

/* Nearest-anchor representation of every key and value vector ("AnchorKV: Anchor-Residual
 * KV Cache Compression", §3.1): for every position i of segment (b, h) and each side
 * (K, V) the anchor slot j whose vector has the largest cosine similarity with x_i (signed;
 * first slot on ties; cosine 0 against a zero vector) and gamma_i = <x_i, a_j> / |a_j|^2,
 * the coefficient of the orthogonal projection of x_i onto span(a_j).  Anchor positions
 * represent themselves (slot = own, gamma = 1).  Dot products run on tcgen05 tensor cores
 * (bf16 inputs, fp32 accumulation); 1/|a_j| in fp32.
 *   p        budget_mode must be KVSEL_BUDGET_ANCHOR (sizes: k anchors per head <= 1024,
 *            else KVSEL_EUNSUPPORTED)
 *   kv       the vectors to represent (the page projects pre-RoPE keys: pass that view)
 *   anchor_k, anchor_v  device bf16 [n_kept][head_dim]: the anchors' rows, as
 *            kvsel_compact writes them for idx/counts/offsets
 *   idx/counts/offsets  device, the anchors as kvsel_select writes them in ANCHOR mode
 *   slot_k, slot_v      device int32 [n_scores]; gamma_k, gamma_v device fp32 [n_scores],
 *            packed like the scores; slots index the segment's anchor list
 *   ws       workspace of kvsel_workspace_size bytes (holds the anchors' inverse norms) */
int kvsel_anchor_project(const kvsel_params* p, const kvsel_kv* kv, const void* anchor_k, const void* anchor_v,
                         const int32_t* idx, const int32_t* counts, const int64_t* offsets, int32_t* slot_k,
                         float* gamma_k, int32_t* slot_v, float* gamma_v, void* ws, size_t ws_bytes, void* stream);

/* AnchorKV compression front end for one layer, enqueued back to back on `stream`:
 * window scoring (s_attn = the pooled SnapKV score), anchor selection (ANCHOR mode,
 * rand_keys: device fp32 [n_scores] i.i.d. uniform keys), gather of the anchor rows into
 * anchor_k / anchor_v, and kvsel_anchor_project.  Arguments as in those calls. */
int kvsel_run_anchors(const kvsel_params* p, const void* q, const kvsel_kv* kv, const float* rand_keys,
                      float* s_attn, int32_t* idx, int32_t* counts, int64_t* offsets, void* anchor_k, void* anchor_v,
                      int32_t* slot_k, float* gamma_k, int32_t* slot_v, float* gamma_v, void* ws, size_t ws_bytes,
                      void* stream);

/* ---- output perturbation of a kept set --------------------------------------------- */

/* Workspace bytes of kvsel_perturbation for these parameters (host-only). */
int kvsel_perturbation_workspace_size(const kvsel_params* p, size_t* bytes);

/* How much a kept set perturbs the attention output of the observation-window queries
 * ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", Definition 3.1, §3.3 Theorems 3.2 and
 * 3.3, App. C.4 Theorem C.1, App. C.5 Table 9).  For window row w of query head (h, g),
 * softmax weights A_i over the keys it sees (causal, scale as in kvsel_score), kept set S
 * of KV head h, kept mass a = sum_{i in S} A_i and projected values v'_i = W_O^(h,g) v_i:
 *   out[b][h][0][g][w] = ||o - ô||_1 with o = sum_i A_i v'_i and ô = sum_{i in S} A_i v'_i / a
 *                        (eviction as a renormalised 0/1 mask on A, Theorem 3.2)
 *   out[b][h][1][g][w] = C - (2 - 1/a) P, C = sum_i A_i ||v'_i||_1, P = sum_{i in S} A_i ||v'_i||_1
 *                        (Theorem 3.3's bound; C when a = 0)
 *   out[b][h][2][g][w] = 2 (1 - a) max_i ||v'_i||_1 over the keys the row sees
 *                        (the relaxed bound that attention-only selection minimises, C.1)
 *   p        window scoring parameters (window > 0, group * window <= 128, group <= 16,
 *            d_model a multiple of 128); value_aware and the budget fields are not read
 *   q, kv    as kvsel_score (V rows past a request's length in the contiguous layout must
 *            hold finite values: they are multiplied by zero)
 *   w_o      device bf16 [d_model][h_kv*group*head_dim]
 *   idx/counts/offsets  device: the kept set per (request, head), as kvsel_select writes it
 *   out      device fp32 [batch][h_kv][3][group][window]
 *   ws       workspace of kvsel_perturbation_workspace_size bytes, 256-byte aligned
 * The logits and the weighted value sums run on tcgen05 (bf16 inputs, fp32 accumulation;
 * the weights enter as bf16 high and low parts); ||v'||_1 uses the value-norm GEMM once
 * per group member; the output projection is fp32 on CUDA cores. */
int kvsel_perturbation(const kvsel_params* p, const void* q, const kvsel_kv* kv, const void* w_o, const int32_t* idx,
                       const int32_t* counts, const int64_t* offsets, float* out, void* ws, size_t ws_bytes,
                       void* stream);

/* Static description of an error code. */
const char* kvsel_strerror(int code);

/* Library version string. */
const char* kvsel_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVSEL_H */
