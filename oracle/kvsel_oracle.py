"""fp64 CPU oracle for end-of-prefill KV scoring, selection and compaction.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg may import or run this module; the product path never does.
It shares no code with the CUDA library (no kernels, headers, helpers or tables): it is
a plain, slow restatement of what the source pages define, in float64 on inputs decoded
exactly from bfloat16, with numpy library primitives (matmul, exp, sort) as steps and no
blocking, fusion or reordering beyond what the definitions state.

Sources (cited by page title and section):
  [CKV]  "CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기" (CriticalKV, Korean
         translation with add-ons): §3.3 Theorem 3.3, §3.4 Algorithm 1 (two-stage greedy
         selection), Algorithm 2 (observation-window scoring), §3.5, §4.1, footnote 3,
         App. C.4 Theorem C.1, App. D.4, and the kvpress notes (section 3 of the add-on).
  [KVZ]  "KVzip: Query-Agnostic KV Cache Compression with Context Reconstruction":
         §2.2 (GQA cache structure), §3.2 (maximum cross-attention score), §3.4 (chunked
         scoring; head-level score as the maximum over the sequence), §3.6 (head-level
         eviction), §4.2 (non-uniform head budget, kept system prompt, eviction on the
         un-replicated cache), §6.5 (softmax-free variant, KVzip-logit), §7.1
         (variable-length decode).
  [VKV]  "VestigeKV: The NoPE-MLA KV Cache Carries Its Own Eviction Signal in a Vestigial
         Branch": §4.1 (4 sinks + recent window are always kept; evicted rows are
         archived, not deleted: kept and archived sides partition the positions).
  [AKV]  "AnchorKV: Anchor-Residual KV Cache Compression": §3.2 (recent window always
         kept; SnapKV pooled scoring).

Readings taken where the pages are silent or garbled (each also listed in the design
notes): logits carry the model's 1/sqrt(d) scale; window queries are causal; average
pooling pads with zeros and divides by k, max pooling ignores out-of-range positions;
the GQA value norm uses the group's summed W_O slice (one D-vector per token and KV
head); forced entries count inside the budget and inside stage 1; budgets round down;
ties order by index ascending.

Every function below has at least one pin in tests/test_oracle_pins.py; none is
"parity unpinned".
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import numpy as np

EPS_DEFAULT = 1e-4    # [CKV] footnote 3: the small constant added before the product
ALPHA_DEFAULT = 0.5   # [CKV] §3.5 / §4.1: first-stage share used in every experiment


# ---------------------------------------------------------------------------------------
# decoding
# ---------------------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (uint16) as float64."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------------------
# scoring: observation window (Algorithm 2, [CKV] §3.4) and query-agnostic ([KVZ] §3.2)
# ---------------------------------------------------------------------------------------
def window_logits(q: np.ndarray, k: np.ndarray, scale: Optional[float] = None,
                  causal: bool = True) -> np.ndarray:
    """Logits of the window queries of one KV head against all of its keys.

    q: [G][W][d] (group heads x window positions), k: [n][d].  Returns l[g][w][i] =
    scale * <q[g][w], k[i]>; with ``causal`` the window row w sits at position n-W+w and
    keys i > n-W+w are masked to -inf (the queries of the last W prompt tokens see only
    their own prefix).  Algorithm 2 forms softmax(Q_hat K^T) with Q_hat the last n'
    queries; the scale is the model's attention scale (reading: 1/sqrt(d)).
    """
    G, W, d = q.shape
    n = k.shape[0]
    if scale is None or scale == 0.0:
        scale = 1.0 / math.sqrt(d)
    l = np.matmul(q.reshape(G * W, d), k.T).reshape(G, W, n) * scale
    if causal:
        pos = n - W + np.arange(W)
        mask = np.arange(n)[None, :] > pos[:, None]          # [W][n]
        l = np.where(mask[None, :, :], -np.inf, l)
    return l


def softmax_rows(l: np.ndarray) -> np.ndarray:
    """Row softmax along the last axis (masked entries -inf give exactly 0)."""
    m = np.max(l, axis=-1, keepdims=True)
    e = np.exp(l - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def reduce_rows(p: np.ndarray, op: str) -> np.ndarray:
    """Reduce attention rows over the group heads and window positions.

    Algorithm 2 averages over the window rows (``A.mean(dim=0)``); the GQA group of a KV
    head shares one score ([KVZ] §2.2, §4.2).  op: "mean" | "sum" | "max".
    """
    rows = p.reshape(-1, p.shape[-1])
    if op == "mean":
        return rows.mean(axis=0)
    if op == "sum":
        return rows.sum(axis=0)
    if op == "max":
        return rows.max(axis=0)
    raise ValueError(op)


def window_scores(q: np.ndarray, k: np.ndarray, reduce: str = "mean",
                  scale: Optional[float] = None, causal: bool = True) -> np.ndarray:
    """s_raw[i]: window attention of key i reduced over (g, w) — Algorithm 2, [CKV]."""
    return reduce_rows(softmax_rows(window_logits(q, k, scale, causal)), reduce)


def pool1d(s: np.ndarray, kind: str, kernel: int) -> np.ndarray:
    """1-D pooling along the sequence, stride 1, output length n (Algorithm 2, SnapKV).

    Window of key i: positions [i - kernel//2, i + kernel//2].  "max" ignores positions
    outside [0, n); "avg" treats them as zeros and divides by ``kernel``.
    """
    n = s.shape[0]
    if kind == "none" or kernel <= 1:
        return s.copy()
    h = kernel // 2
    if kind == "max":
        padded = np.concatenate([np.full(h, -np.inf), s, np.full(h, -np.inf)])
        return np.lib.stride_tricks.sliding_window_view(padded, 2 * h + 1).max(axis=-1)
    if kind == "avg":
        padded = np.concatenate([np.zeros(h), s, np.zeros(h)])
        return np.lib.stride_tricks.sliding_window_view(padded, 2 * h + 1).sum(axis=-1) / kernel
    raise ValueError(kind)


def wo_slices(w_o: np.ndarray, h: int, group: int, d: int) -> List[np.ndarray]:
    """The D x d output-projection slices of the query heads sharing KV head h.

    W_O is stored as an nn.Linear weight [D][H_q*d]; query head q = h*G + g owns the
    input columns [q*d, (q+1)*d).
    """
    return [w_o[:, (h * group + g) * d:(h * group + g + 1) * d] for g in range(group)]


def value_norm(v: np.ndarray, w_o: np.ndarray, h: int, group: int,
               mode: str = "group_sum", row_block: int = 4096, norm: str = "l1") -> np.ndarray:
    """nu[i] = L1 norm of the value state v[i] projected through W_O ([CKV] Algorithm 1,
    Theorem 3.3; kvpress notes: L1 norm of V @ Wo[head]); with norm="l2" the Euclidean
    norm, the other distance [CKV] App. C.3 compares (reading of the garbled symbols:
    the paper adopts L1 for simplicity and reports L2 as giving similar gains).

    v: [n][d] values of KV head h.  GQA reading ("group_sum", default): the value is
    replicated over the G query heads of the group, so its projected contribution is
    (sum_g W_O^(h,g)) v — one D-vector per token and KV head, which is the intermediate
    whose size App. D.4 quotes.  "per_head": sum_g ||W_O^(h,g) v||_1 (upper bound).
    Rows are processed in blocks only to bound memory; each row is independent.
    """
    n, d = v.shape
    sl = wo_slices(w_o, h, group, d)
    out = np.empty(n)
    if norm == "l1":
        def rownorm(x):
            return np.abs(x).sum(axis=1)
    elif norm == "l2":
        def rownorm(x):
            return np.sqrt((x * x).sum(axis=1))
    else:
        raise ValueError(norm)
    if mode == "group_sum":
        wbar = np.zeros_like(sl[0])
        for s in sl:
            wbar = wbar + s
        for a in range(0, n, row_block):
            out[a:a + row_block] = rownorm(v[a:a + row_block] @ wbar.T)
    elif mode == "per_head":
        out[:] = 0.0
        for s in sl:
            for a in range(0, n, row_block):
                out[a:a + row_block] += rownorm(v[a:a + row_block] @ s.T)
    else:
        raise ValueError(mode)
    return out


def combine(s_pool: np.ndarray, nu: np.ndarray, eps: float = EPS_DEFAULT) -> np.ndarray:
    """Value-aware criterion (A + eps) * nu — [CKV] Algorithm 1; eps from footnote 3."""
    return (s_pool + eps) * nu


def query_agnostic_scores(q: np.ndarray, k: np.ndarray, scale: Optional[float] = None,
                          q_chunk: int = 0) -> np.ndarray:
    """KVzip maximum cross-attention score of every key ([KVZ] §3.2).

    q: [G][m][d] query features of one KV head, k: [n][d].  S[i] = max over group heads
    g and query positions j of softmax_i(q[g][j] . k / sqrt(d)).  Softmax runs over all
    n keys, without a causal mask.  Query positions may be processed in chunks of
    ``q_chunk`` and combined with max, as [KVZ] §3.4 aggregates chunk scores.
    """
    G, m, d = q.shape
    if scale is None or scale == 0.0:
        scale = 1.0 / math.sqrt(d)
    step = m if q_chunk <= 0 else q_chunk
    S = np.zeros(k.shape[0])
    for a in range(0, m, step):
        qa = q[:, a:a + step, :].reshape(-1, d)
        p = softmax_rows((qa @ k.T) * scale)
        S = np.maximum(S, p.max(axis=0))
    return S


def query_agnostic_logit_scores(q: np.ndarray, k: np.ndarray, scale: Optional[float] = None,
                                q_chunk: int = 0) -> np.ndarray:
    """KVzip-logit, the softmax-free variant ([KVZ] §6.5): S[i] = max over group heads g
    and query positions j of the scaled dot product q[g][j] . k[i] / sqrt(d) itself,
    without softmax normalisation.  Chunks combine with max as in §3.4."""
    G, m, d = q.shape
    if scale is None or scale == 0.0:
        scale = 1.0 / math.sqrt(d)
    step = m if q_chunk <= 0 else q_chunk
    S = np.full(k.shape[0], -np.inf)
    for a in range(0, m, step):
        qa = q[:, a:a + step, :].reshape(-1, d)
        S = np.maximum(S, ((qa @ k.T) * scale).max(axis=0))
    return S


def head_scores(S: np.ndarray) -> np.ndarray:
    """Head-level importance ([KVZ] §3.4, §3.6): S_head = max over the sequence of the
    per-key score of that head.  S: [H][n] -> [H]."""
    return S.max(axis=1)


# ---------------------------------------------------------------------------------------
# forced entries and selection
# ---------------------------------------------------------------------------------------
def forced_mask(n: int, n_sink: int, n_recent: int) -> np.ndarray:
    """Attention sinks [0, n_sink) and the recent window [n-n_recent, n) are always kept
    ([VKV] §4.1; [AKV] §3.2; [CKV] kvpress notes: stage-1 picks kept via the max value)."""
    f = np.zeros(n, dtype=bool)
    f[:min(n_sink, n)] = True
    if n_recent > 0:
        f[max(n - n_recent, 0):] = True
    return f


def top_b(scores: np.ndarray, budget: int, forced: np.ndarray) -> np.ndarray:
    """Indices (ascending) of the top ``budget`` entries: forced entries first, then by
    score descending, ties by index ascending.  Top_k of [CKV] Algorithm 1/2."""
    n = scores.shape[0]
    nf = int(forced.sum())
    if budget < nf or budget > n:
        raise ValueError(f"budget {budget} outside [{nf}, {n}]")
    key = np.where(forced, np.inf, scores)
    order = np.lexsort((np.arange(n), -key))  # primary: key descending; then index
    return np.sort(order[:budget]).astype(np.int64)


def select_two_stage(s_pool: np.ndarray, s_val: np.ndarray, budget: int,
                     forced: np.ndarray, alpha: float = ALPHA_DEFAULT) -> np.ndarray:
    """[CKV] Algorithm 1: stage 1 keeps b' = floor(alpha*b) entries by attention score
    (forced entries inside it), stage 2 fills the remaining b - |S1| by the value-aware
    criterion among the entries not yet kept."""
    b1 = int(math.floor(alpha * budget))
    nf = int(forced.sum())
    s1 = top_b(s_pool, max(b1, nf), forced)
    keep1 = np.zeros_like(forced)
    keep1[s1] = True
    return top_b(s_val, budget, keep1)


def head_budget(n: int, ratio: float) -> int:
    return int(math.floor(ratio * n))


def select_per_layer(scores: np.ndarray, budget: int, forced: np.ndarray,
                     floor_per_head: int) -> List[np.ndarray]:
    """One budget shared by all heads of a layer (AdaKV / [KVZ] §4.2 non-uniform head
    budget): keep the top entries over the flattened [H][n] scores.

    Reading for the per-head floor: every head first keeps its forced entries plus its
    own top entries up to ``floor_per_head``; the remaining slots go to a flattened
    top over all heads' other entries, ties by flat index h*n + i ascending.
    """
    H, n = scores.shape
    keep = np.zeros((H, n), dtype=bool)
    for h in range(H):
        nf = int(forced[h].sum())
        keep[h, top_b(scores[h], min(max(floor_per_head, nf), n), forced[h])] = True
    if budget < int(keep.sum()) or budget > H * n:
        raise ValueError("layer budget below the floors or above H*n")
    flat = top_b(scores.reshape(-1), budget, keep.reshape(-1))
    return [flat[(flat >= h * n) & (flat < (h + 1) * n)] - h * n for h in range(H)]


def select_two_stage_per_layer(s_pool: np.ndarray, s_val: np.ndarray, budget: int, forced: np.ndarray,
                               floor_per_head: int, alpha: float = ALPHA_DEFAULT) -> List[np.ndarray]:
    """Value-aware selection under one budget per layer ([CKV] §3.4 Algorithm 2: line 1
    allocates the layer's budget across heads, AdaKV-style; line 8 then runs Algorithm 1
    per head).  Reading: head h's budget b_h is the number of its entries in the layer-wide
    top-``budget`` of the pooled attention score (with the per-head floor, as in
    select_per_layer); each head then keeps b_h entries by the two-stage criterion."""
    alloc = select_per_layer(s_pool, budget, forced, floor_per_head)
    return [select_two_stage(s_pool[h], s_val[h], len(alloc[h]), forced[h], alpha)
            for h in range(s_pool.shape[0])]


# ---------------------------------------------------------------------------------------
# compaction
# ---------------------------------------------------------------------------------------
def compact(x: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Kept rows of one KV head's cache in index order ([KVZ] §4.2: eviction acts on the
    un-replicated KV head; §7.1: per-head variable-length result)."""
    return x[np.asarray(idx, dtype=np.int64)]


def partition(n: int, idx: np.ndarray):
    """Kept positions and their complement, the evicted ones, both ascending ([VKV] §4.1:
    eviction moves rows from the hot cache to an archive and deletes nothing, so every
    position of [0, n) is in exactly one of the two sets)."""
    kept = np.zeros(n, dtype=bool)
    kept[np.asarray(idx, dtype=np.int64)] = True
    return np.flatnonzero(kept), np.flatnonzero(~kept)


def archive(x: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Evicted rows of one KV head's cache in index order ([VKV] §4.1: the archive side of
    the partition, bit-exact)."""
    return x[partition(x.shape[0], idx)[1]]


def unpage(pool: np.ndarray, table: np.ndarray, n: int) -> np.ndarray:
    """[H][n][d] view of one request held in a block pool [blocks][bs][H][d]."""
    bs = pool.shape[1]
    rows = [pool[table[i // bs], i % bs] for i in range(n)]  # each [H][d]
    return np.stack(rows, axis=1) if n else np.zeros((pool.shape[2], 0, pool.shape[3]), pool.dtype)


# ---------------------------------------------------------------------------------------
# one layer, end to end
# ---------------------------------------------------------------------------------------
def run_layer(q_bits: np.ndarray, k_bits: Sequence[np.ndarray], v_bits: Sequence[np.ndarray],
              w_o_bits: Optional[np.ndarray], *, group: int, window: int, causal: bool,
              reduce: str, pool: str, pool_kernel: int, value_aware: bool, eps: float,
              alpha: float, n_sink: int, n_recent: int, budget_mode: str,
              budget_ratio: float, floor_ratio: float = 0.0, scale: Optional[float] = None,
              q_chunk: int = 0, wo_mode: str = "group_sum", heads: Optional[Sequence[int]] = None,
              compact_out: bool = True, value_norm_kind: str = "l1") -> List[dict]:
    """Score -> select -> compact for every request of one layer.

    q_bits: [B][H][G][W][d] bf16 bits (W = n for query-agnostic scoring), k_bits/v_bits:
    per request [H][n][d] bf16 bits, w_o_bits: [D][H*G*d] bf16 bits or None.
    Returns one dict per request with float64 s_raw, s_pool, nu, s_val ([H][n]) and the
    kept indices (list over heads), plus the compacted K/V bits when ``compact_out``.
    """
    B = len(k_bits)
    out = []
    w_o = bf16_to_f64(w_o_bits) if value_aware else None
    for b in range(B):
        k = bf16_to_f64(k_bits[b])
        H, n, d = k.shape
        hs = range(H) if heads is None else heads
        s_raw = np.zeros((H, n))
        for h in hs:
            qh = bf16_to_f64(q_bits[b][h])
            if window > 0:
                s_raw[h] = window_scores(qh, k[h], reduce, scale, causal)
            elif reduce == "max_logit":
                s_raw[h] = query_agnostic_logit_scores(qh, k[h], scale, q_chunk)
            else:
                s_raw[h] = query_agnostic_scores(qh, k[h], scale, q_chunk)
        s_pool = np.stack([pool1d(s_raw[h], pool, pool_kernel) for h in range(H)])
        nu = s_val = None
        if value_aware:
            v = bf16_to_f64(v_bits[b])
            nu = np.zeros((H, n))
            for h in hs:
                nu[h] = value_norm(v[h], w_o, h, group, wo_mode, norm=value_norm_kind)
            s_val = combine(s_pool, nu, eps)
        fm = forced_mask(n, n_sink, n_recent)
        if budget_mode == "head":
            bh = head_budget(n, budget_ratio)
            if value_aware:
                idx = [select_two_stage(s_pool[h], s_val[h], bh, fm, alpha) for h in range(H)]
            else:
                idx = [top_b(s_pool[h], bh, fm) for h in range(H)]
        elif budget_mode == "layer":
            bl = int(math.floor(budget_ratio * n * H))
            fl = int(math.floor(floor_ratio * n))
            if value_aware:
                idx = select_two_stage_per_layer(s_pool, s_val, bl, np.stack([fm] * H), fl, alpha)
            else:
                idx = select_per_layer(s_pool, bl, np.stack([fm] * H), fl)
        else:
            raise ValueError(budget_mode)
        r = dict(n=n, s_raw=s_raw, s_pool=s_pool, nu=nu, s_val=s_val, idx=idx)
        if compact_out:
            r["k_out"] = [compact(k_bits[b][h], idx[h]) for h in range(H)]
            r["v_out"] = [compact(v_bits[b][h], idx[h]) for h in range(H)]
        out.append(r)
    return out


def run_workload_layer(wl, inputs: dict, **kw) -> List[dict]:
    """run_layer with the choices of a datagen.Workload."""
    return run_layer(inputs["q"], inputs["k"], inputs["v"], inputs["w_o"], group=wl.group,
                     window=wl.window, causal=wl.causal, reduce=wl.reduce, pool=wl.pool,
                     pool_kernel=wl.pool_kernel, value_aware=wl.value_aware, eps=wl.eps,
                     alpha=wl.alpha, n_sink=wl.n_sink, n_recent=wl.n_recent,
                     budget_mode=wl.budget_mode, budget_ratio=wl.budget_ratio,
                     floor_ratio=wl.floor_ratio, q_chunk=wl.q_chunk,
                     value_norm_kind=wl.value_norm, **kw)
