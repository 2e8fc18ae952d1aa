"""Seeded synthetic inputs for end-of-prefill KV scoring, selection and compaction.

This module is shared by the tests, the benchmark and the oracle's callers.  It holds
none of the method's arithmetic: only the workload table (shapes, budgets, pooling
choices), the seeds, and the value distributions of the synthetic Q/K/V/W_O tensors.
Every tensor is produced in float32 from ``numpy.random.Generator(PCG64)`` streams and
rounded to bfloat16 (round to nearest, ties to even); bfloat16 data is handed out as
``numpy.uint16`` bit patterns so that both the CUDA path and the fp64 oracle decode the
same bits.

The workloads stand in for the pages' evaluation suites (Ruler, LongBench, SCBench,
SQuAD, GSM8K, needle-in-a-haystack) and trained models, none of which are available:
shapes follow Llama-3.1-8B (8 KV heads, group 4), Qwen2.5-7B (4 KV heads, group 7) and
Llama-3.1-70B (8 KV heads, group 8), the observation window of 32 and pooling kernel 7
used by SnapKV/AdaKV in CriticalKV §4.1, and KVzip's 2K query chunks (KVzip §3.4).

Random streams are split into fixed chunks of 2**22 values, each with its own
``SeedSequence([seed, tensor_tag, chunk])``, so the result does not depend on how many
threads fill them.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional

import numpy as np

_CHUNK = 1 << 22
_THREADS = 16

# tensor tags inside one layer's seed
_TAG_Q, _TAG_K, _TAG_V, _TAG_WO, _TAG_KSCALE, _TAG_HEAVY, _TAG_CTX, _TAG_BLOCKS, _TAG_RAND = range(9)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: model shape, scoring choices and budget."""

    cid: int
    name: str
    layers: int
    h_kv: int
    group: int
    head_dim: int
    d_model: int          # rows of W_O (output features); only used when value_aware
    n_ctx: int            # context length (max length for the ragged batch)
    window: int           # observation-window queries per group head; 0 = all n positions
    causal: bool
    reduce: str           # "sum" | "mean" | "max" | "max_logit" (query-agnostic, no softmax)
    pool: str             # "none" | "max" | "avg"
    pool_kernel: int
    value_aware: bool
    alpha: float
    eps: float
    n_sink: int
    n_recent: int
    budget_mode: str      # "head" | "layer" | "anchor" (k = budget_ratio*n anchors, rho = alpha)
    budget_ratio: float
    floor_ratio: float
    batch: int = 1
    n_min: int = 0        # ragged batch: contexts drawn uniformly from [n_min, n_ctx]
    paged: bool = False
    block_size: int = 16
    q_chunk: int = 0      # query-agnostic scoring: query rows per chunk (per group head)
    key_structure: str = "plain"  # "heavy" | "lognormal" | "zipf" | "plain"
    value_norm: str = "l1"        # value-aware: "l1" (default) | "l2" (norm of W_h v)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def rows_per_head(self) -> int:
        return self.group * (self.window if self.window > 0 else self.n_ctx)


# The five workloads.  Budgets, pooling and forced entries follow the pages where they
# are stated (window 32 / maxpool 7: CriticalKV §4.1; alpha 0.5: CriticalKV §3.5;
# eps 1e-4: CriticalKV footnote 3; 4 sinks + recent window: VestigeKV §4.1; KVzip
# per-layer budget across heads: KVzip §4.2) and are the builder's reading elsewhere.
WORKLOADS: Dict[int, Workload] = {
    1: Workload(1, "llama8b-layer-4k", 1, 8, 4, 128, 4096, 4096, 32, True, "sum", "max", 7,
                False, 0.5, 1e-4, 4, 32, "head", 0.2, 0.0, key_structure="heavy"),
    2: Workload(2, "llama3.1-8b-32k-stack", 32, 8, 4, 128, 4096, 32768, 32, True, "mean", "avg", 5,
                True, 0.5, 1e-4, 4, 32, "head", 0.4, 0.0, key_structure="lognormal"),
    3: Workload(3, "qwen2.5-7b-128k-stack", 28, 4, 7, 128, 3584, 131072, 64, True, "mean", "max", 7,
                False, 0.5, 1e-4, 4, 64, "layer", 0.1, 0.05, key_structure="zipf"),
    4: Workload(4, "ragged-paged-batch16", 1, 8, 4, 128, 4096, 65536, 32, True, "mean", "avg", 5,
                True, 0.5, 1e-4, 4, 32, "head", 0.25, 0.0, batch=16, n_min=2048, paged=True,
                block_size=16, key_structure="plain"),
    5: Workload(5, "llama3.1-70b-query-agnostic-32k", 1, 8, 8, 128, 8192, 32768, 0, False, "max", "none", 1,
                False, 0.5, 1e-4, 4, 0, "layer", 0.3, 0.0, q_chunk=2048, key_structure="plain"),
    # AnchorKV anchor selection and nearest-anchor projection on the Llama-3.1-8B 32K
    # shape: W = 32, k = n/128 anchors, rho = 0.7 (carried in alpha), kappa = 7 (AnchorKV
    # §4.1); the recent window is the only forced set (§3.2).
    6: Workload(6, "llama3.1-8b-32k-anchors", 1, 8, 4, 128, 4096, 32768, 32, True, "mean", "max", 7,
                False, 0.7, 1e-4, 0, 32, "anchor", 1.0 / 128, 0.0, key_structure="lognormal"),
}


def layer_seed(cid: int, layer: int) -> int:
    return 1234 + cid * 1000 + layer


def _normal_f32(seed: int, tag: int, n: int, threads: int = _THREADS) -> np.ndarray:
    out = np.empty(n, np.float32)
    nch = (n + _CHUNK - 1) // _CHUNK

    def fill(j: int) -> None:
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, j])))
        s = j * _CHUNK
        e = min(n, s + _CHUNK)
        g.standard_normal(e - s, dtype=np.float32, out=out[s:e])

    if nch == 1 or threads <= 1:
        for j in range(nch):
            fill(j)
    else:
        with ThreadPoolExecutor(min(threads, nch)) as ex:
            list(ex.map(fill, range(nch)))
    return out


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    try:
        import torch

        return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover - numpy path, same rounding
        u = x.view(np.uint32).astype(np.uint64)
        r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        return r.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def context_lengths(wl: Workload, layer: int = 0) -> List[int]:
    """Per-request context lengths (one entry unless the workload is a ragged batch)."""
    if wl.batch == 1 or wl.n_min <= 0:
        return [wl.n_ctx] * wl.batch
    g = _rng(layer_seed(wl.cid, 0), _TAG_CTX)
    return [int(v) for v in g.integers(wl.n_min, wl.n_ctx + 1, size=wl.batch)]


def make_layer(wl: Workload, layer: int = 0, n_ctx: Optional[int] = None,
               threads: int = _THREADS) -> dict:
    """Synthetic inputs of one layer.

    Returns a dict of numpy arrays (bf16 as uint16 bits):
      q      : [B][H][G][W][d]   observation-window queries (W = n for query-agnostic scoring)
      k, v   : list over requests of [H][n_b][d]
      w_o    : [D][H*G*d]        (value-aware workloads only, else None)
      n_ctx  : list of per-request lengths
      paged  : dict(k_pool, v_pool [num_blocks][block][H][d], block_table [B][max_blocks])
               when the workload is paged
      rand   : list over requests of [H][n_b] float32 i.i.d. uniform [0, 1) keys (anchor
               workloads: the random share of the anchors takes the largest keys)
    ``n_ctx`` overrides the context length (single-request workloads only), which the
    tests use for smaller cases of the same recipe.
    """
    seed = layer_seed(wl.cid, layer)
    H, G, d = wl.h_kv, wl.group, wl.head_dim
    if n_ctx is not None:
        assert wl.batch == 1
        lens = [int(n_ctx)]
    else:
        lens = context_lengths(wl, layer)
    W = wl.window if wl.window > 0 else None
    B = len(lens)

    qs, ks, vs, rs = [], [], [], []
    for b, n in enumerate(lens):
        rows = W if W is not None else n
        sub = seed * 64 + b
        q = _normal_f32(sub, _TAG_Q, H * G * rows * d, threads).reshape(H, G, rows, d)
        q = to_bf16_bits(q)
        k = _normal_f32(sub, _TAG_K, H * n * d, threads).reshape(H, n, d)
        if wl.key_structure == "heavy":
            # 64 heavy-hitter keys per head: 4*sqrt(d) along the unit mean window query
            # of the group, plus N(0,1) noise (the noise is the key's own draw).
            g = _rng(sub, _TAG_HEAVY)
            qf = bf16_bits_to_f32(q)
            hi = max(wl.n_sink, 0)
            lo_end = n - (W or 0)
            for h in range(H):
                u = qf[h].reshape(-1, d).mean(axis=0)
                u = u / np.linalg.norm(u)
                cnt = min(64, max(lo_end - hi, 0))
                pos = g.choice(np.arange(hi, lo_end), size=cnt, replace=False)
                k[h, pos, :] += (4.0 * math.sqrt(d)) * u[None, :]
        elif wl.key_structure == "lognormal":
            xi = _normal_f32(sub, _TAG_KSCALE, n, 1)
            k *= np.exp(0.5 * xi)[None, :, None]
        elif wl.key_structure == "zipf":
            g = _rng(sub, _TAG_KSCALE)
            m = np.minimum(g.zipf(1.1, size=n), 8).astype(np.float32)
            k *= m[None, :, None]
        ks.append(to_bf16_bits(k))
        vs.append(to_bf16_bits(_normal_f32(sub, _TAG_V, H * n * d, threads).reshape(H, n, d)))
        qs.append(q)
        if wl.budget_mode == "anchor":
            rs.append(_rng(sub, _TAG_RAND).random((H, n), dtype=np.float32))

    out = dict(q=np.stack(qs) if W is not None else qs[0][None], k=ks, v=vs, n_ctx=lens, w_o=None,
               paged=None, rand=rs if wl.budget_mode == "anchor" else None)
    if wl.value_aware:
        D = wl.d_model
        w = _normal_f32(seed, _TAG_WO, D * H * G * d, threads) * np.float32(0.02)
        out["w_o"] = to_bf16_bits(w.reshape(D, H * G * d))
    if wl.paged:
        out["paged"] = make_paged(ks, vs, wl.block_size, _rng(seed, _TAG_BLOCKS))
    return out


def make_paged(ks: List[np.ndarray], vs: List[np.ndarray], block: int,
               g: np.random.Generator) -> dict:
    """Scatter per-request [H][n][d] caches into a shuffled block pool.

    Pool layout [num_blocks][block][H][d]; block_table[b][j] is the physical block that
    holds tokens [j*block, (j+1)*block) of request b (-1 past the end).  Physical blocks
    are a random permutation over all requests' blocks; slots past a request's end are
    left as zeros.
    """
    H, d = ks[0].shape[0], ks[0].shape[2]
    nblk = [(k.shape[1] + block - 1) // block for k in ks]
    total = int(sum(nblk))
    perm = g.permutation(total).astype(np.int32)
    maxb = max(nblk)
    table = np.full((len(ks), maxb), -1, np.int32)
    kp = np.zeros((total, block, H, d), np.uint16)
    vp = np.zeros((total, block, H, d), np.uint16)
    c = 0
    for b, (k, v) in enumerate(zip(ks, vs)):
        n = k.shape[1]
        for j in range(nblk[b]):
            p = perm[c]
            c += 1
            table[b, j] = p
            s, e = j * block, min(n, (j + 1) * block)
            kp[p, : e - s] = k[:, s:e, :].transpose(1, 0, 2)
            vp[p, : e - s] = v[:, s:e, :].transpose(1, 0, 2)
    return dict(k_pool=kp, v_pool=vp, block_table=table, block_size=block)


def anchor_keys(h_kv: int, n: int, seed: int) -> np.ndarray:
    """[H][n] float32 i.i.d. uniform [0, 1) keys for the random share of the anchors."""
    return _rng(seed, _TAG_RAND).random((h_kv, n), dtype=np.float32)


def anchor_positions(n: int, k: int, n_recent: int, seed: int) -> np.ndarray:
    """A given anchor list for projection-only tests: the recent window plus
    k - |window| distinct positions drawn uniformly from the rest, ascending (int32)."""
    nr = min(n_recent, n, k)
    rest = _rng(seed, _TAG_RAND).choice(n - nr, size=k - nr, replace=False) if k > nr else np.zeros(0, np.int64)
    return np.sort(np.concatenate([rest, np.arange(n - nr, n)])).astype(np.int32)


def random_scores(n_rows: int, n: int, seed: int, tie_frac: float = 0.1) -> np.ndarray:
    """Non-negative float32 score rows with planted exact ties (for selection-only tests).

    A fraction ``tie_frac`` of entries copies a value from elsewhere in the row, so equal
    keys straddle the selection threshold; values span several binades.
    """
    g = _rng(seed, 99)
    s = np.exp(g.standard_normal((n_rows, n)) * 3.0).astype(np.float32)
    ntie = int(tie_frac * n)
    for r in range(n_rows):
        src = g.integers(0, n, size=max(ntie // 8, 1))
        dst = g.integers(0, n, size=ntie)
        s[r, dst] = s[r, src[g.integers(0, len(src), size=ntie)]]
    return s


def random_sorted_indices(n: int, counts: List[int], seed: int) -> List[np.ndarray]:
    """Ascending distinct index sets in [0, n) with the given sizes (compaction tests)."""
    g = _rng(seed, 98)
    return [np.sort(g.choice(n, size=c, replace=False)).astype(np.int32) for c in counts]
