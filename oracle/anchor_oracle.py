"""fp64 CPU oracle for AnchorKV anchor selection and nearest-anchor projection.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg may import or run this module; the product path never does.
It shares no code with the CUDA library.  Source:

  [AKV]  "AnchorKV: Anchor-Residual KV Cache Compression":
         §3.1 (anchor-residual representation: every vector is projected orthogonally onto
              the span of the one anchor with the largest cosine similarity and stored as
              that anchor's index and the scalar coefficient gamma),
         §3.2 (anchor selection per KV head: the recent W positions are always stored
              exactly and count inside the anchor budget; of the remaining slots a share
              rho goes to the highest SnapKV-pooled attention scores, the rest is drawn
              uniformly at random over the context),
         §4.1 (fixed settings: W = 32, k = S/128 anchors, rho = 0.7, kappa = 7).

Readings where the page is silent (also listed in the design notes):
  * k = floor(n / 128), but never fewer than the forced entries (the recent window
    counts inside k) and never more than n.
  * The score share is floor(rho * (k - |F|)); the random share is the rest.
  * "Uniformly at random over the context" draws without replacement from the positions
    not already chosen.  The random draw is an input: one i.i.d. uniform key per
    position, and the draw takes the largest keys (ties by index ascending), which is a
    uniform sample without replacement.
  * Cosine similarity is signed (the anchor with the largest cosine, not the largest
    |cosine|); the cosine with a zero vector is 0; ties go to the lowest anchor slot.
  * Anchor positions represent themselves: slot = their own, gamma = 1.
  * The keys scored and the keys projected are the same synthetic tensor (the page
    scores post-RoPE keys and projects pre-RoPE keys; synthetic keys carry no RoPE).

Every function has pins in tests/test_oracle_pins.py; none is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import List, Optional

import numpy as np

from .kvsel_oracle import bf16_to_f64, forced_mask, pool1d, top_b, window_scores

RHO_DEFAULT = 0.7      # [AKV] §4.1
ANCHOR_DIV = 128       # [AKV] §4.1: k = S / 128


def anchor_count(n: int, n_forced: int, div: int = ANCHOR_DIV) -> int:
    """Anchors of one KV head with n positions ([AKV] §4.1 k = S/128; §3.2: the recent
    window is part of the anchor budget)."""
    return min(n, max(n // div, n_forced))


def select_anchors(s_pool: np.ndarray, rand_key: np.ndarray, k: int, forced: np.ndarray,
                   rho: float = RHO_DEFAULT) -> np.ndarray:
    """Anchor positions of one KV head, ascending ([AKV] §3.2).

    The forced entries (recent window) come first; floor(rho * (k - |F|)) further
    positions by pooled attention score (descending, ties by index); the remaining
    k - |S1| positions are a uniform draw over the rest, realised as the largest
    ``rand_key`` values (descending, ties by index).
    """
    nf = int(forced.sum())
    k1 = nf + int(math.floor(rho * (k - nf)))
    s1 = top_b(s_pool, k1, forced)
    keep1 = np.zeros_like(forced)
    keep1[s1] = True
    return top_b(rand_key, k, keep1)


def anchor_project(x: np.ndarray, anchors: np.ndarray):
    """Nearest-anchor representation of every vector of one KV head ([AKV] §3.1).

    x: [n][d] float64, anchors: ascending positions [k].  For each position i the anchor
    slot j maximising cos(x_i, x_{a_j}) (first slot on ties; cosine 0 against a zero
    vector) and gamma_i = <x_i, a_j> / <a_j, a_j>, the coefficient of the orthogonal
    projection onto span(a_j) (0 for a zero anchor).  Anchor positions get their own slot
    and gamma = 1.  Returns (slot int64 [n], gamma float64 [n], cos float64 [n][k]).
    """
    anchors = np.asarray(anchors, dtype=np.int64)
    A = x[anchors]                                   # [k][d]
    dots = x @ A.T                                   # [n][k]
    an = np.sqrt(np.einsum("kd,kd->k", A, A))
    xn = np.sqrt(np.einsum("nd,nd->n", x, x))
    den = xn[:, None] * an[None, :]
    cos = np.divide(dots, den, out=np.zeros_like(dots), where=den > 0)
    slot = np.argmax(cos, axis=1).astype(np.int64) if len(anchors) else np.zeros(len(x), np.int64)
    a2 = an[slot] ** 2 if len(anchors) else np.zeros(len(x))
    dsel = dots[np.arange(len(x)), slot] if len(anchors) else np.zeros(len(x))
    gamma = np.divide(dsel, a2, out=np.zeros(len(x)), where=a2 > 0)
    slot[anchors] = np.arange(len(anchors))
    gamma[anchors] = 1.0
    return slot, gamma, cos


def run_anchor_layer(q_bits: np.ndarray, k_bits, v_bits, rand, *, window: int, causal: bool,
                     reduce: str, pool: str, pool_kernel: int, n_sink: int, n_recent: int,
                     rho: float = RHO_DEFAULT, div: int = ANCHOR_DIV, scale: Optional[float] = None,
                     heads=None, project: bool = True) -> List[dict]:
    """Anchor selection and projection for every request of one layer ([AKV] §3.1-§3.2).

    q_bits [B][H][G][W][d], k_bits / v_bits per request [H][n][d] (bf16 bits), rand per
    request [H][n] float32 uniform keys.  Per request: s_pool [H][n], anchors (list over
    heads) and, with ``project``, slot_k / gamma_k / slot_v / gamma_v [H][n] plus the
    cosine matrices (lists over heads) for tolerance checks.
    """
    out = []
    for b in range(len(k_bits)):
        k = bf16_to_f64(k_bits[b])
        H, n, d = k.shape
        hs = range(H) if heads is None else heads
        s_pool = np.zeros((H, n))
        fm = forced_mask(n, n_sink, n_recent)
        kk = anchor_count(n, int(fm.sum()), div)
        anchors = [None] * H
        for h in hs:
            s_raw = window_scores(bf16_to_f64(q_bits[b][h]), k[h], reduce, scale, causal)
            s_pool[h] = pool1d(s_raw, pool, pool_kernel)
            anchors[h] = select_anchors(s_pool[h], np.asarray(rand[b][h], np.float64), kk, fm, rho)
        r = dict(n=n, k=kk, s_pool=s_pool, anchors=anchors)
        if project:
            v = bf16_to_f64(v_bits[b])
            for side, x in (("k", k), ("v", v)):
                sl = np.zeros((H, n), np.int64)
                ga = np.zeros((H, n))
                cs = [None] * H
                for h in hs:
                    sl[h], ga[h], cs[h] = anchor_project(x[h], anchors[h])
                r["slot_" + side], r["gamma_" + side], r["cos_" + side] = sl, ga, cs
        out.append(r)
    return out


def run_anchor_workload_layer(wl, inputs: dict, **kw) -> List[dict]:
    """run_anchor_layer with the choices of a datagen.Workload (budget_mode "anchor")."""
    return run_anchor_layer(inputs["q"], inputs["k"], inputs["v"], inputs["rand"], window=wl.window,
                            causal=wl.causal, reduce=wl.reduce, pool=wl.pool,
                            pool_kernel=wl.pool_kernel, n_sink=wl.n_sink, n_recent=wl.n_recent,
                            rho=wl.alpha, div=int(round(1.0 / wl.budget_ratio)), **kw)
