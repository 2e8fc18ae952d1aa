"""fp64 CPU oracle for the output perturbation of a kept set (CriticalKV Theorems 3.2, 3.3, C.1).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg may import or run this module; the product path never does.
It shares no code with the CUDA library.  Source:

  [CKV]  "CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기":
         §3.1 (one attention head: weights A over the cached keys, output W_O (A V)),
         Definition 3.1 (the perturbation of the attention output, measured in L1),
         §3.3 Theorem 3.2 (eviction as a multiplicative 0/1 mask N on A, renormalised:
              Â = A ⊙ N / ||A ⊙ N||_1), Theorem 3.3 (the upper bound θ of ||o - ô||_1),
         App. C.4 Theorem C.1 (the relaxed bound that attention-only selection minimises),
         App. C.5 Table 9 (actual perturbation vs both bounds, averaged per layer).

The formulas on the page are lost in extraction; they are restated here from the
mathematics they describe (readings listed in the design notes):
  * For one query row of query head (h, g): v'_i = W_O^(h,g) v_i (the D-dim projected
    value), o = Σ_i A_i v'_i, ô = Σ_i Â_i v'_i, actual = ||o - ô||_1.
  * With a = Σ_{i∈S} A_i (the kept mass), C = Σ_i A_i ||v'_i||_1 and
    P = Σ_{i∈S} A_i ||v'_i||_1, the triangle inequality on
    o - ô = Σ_{i∉S} A_i v'_i - (1/a - 1) Σ_{i∈S} A_i v'_i gives θ = C - (2 - 1/a) P.
  * Bounding every ||v'_i||_1 by the largest one gives θ' = 2 (1 - a) max_i ||v'_i||_1;
    attention-only selection (the largest A_i) minimises it.
  * The query rows are the observation window (the last W prompt positions, causal, the
    model's 1/sqrt(d) scale, as in the scoring oracle); the maximum in θ' runs over the
    keys the row sees.  The kept set S is per KV head, shared by its G query heads.

Every function has pins in tests/test_oracle_pins.py; none is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

from .kvsel_oracle import bf16_to_f64, softmax_rows, window_logits


def attention_rows(q: np.ndarray, k: np.ndarray, scale: Optional[float] = None,
                   causal: bool = True) -> np.ndarray:
    """A[g][w][i]: softmax weights of the window rows of one KV head ([CKV] §3.1)."""
    return softmax_rows(window_logits(q, k, scale, causal))


def masked_weights(A: np.ndarray, keep: np.ndarray) -> np.ndarray:
    """Â = A ⊙ N / ||A ⊙ N||_1 per row ([CKV] Theorem 3.2); keep: bool [n]."""
    AN = A * keep[None, :]
    return AN / AN.sum(axis=1, keepdims=True)


def perturbation_rows(A: np.ndarray, vproj: np.ndarray, keep: np.ndarray):
    """For rows A [R][n] of one query head and projected values vproj [n][D]:
    (actual ||o - ô||_1, bound θ, relaxed bound θ') per row ([CKV] Definition 3.1,
    Theorems 3.2, 3.3, C.1).  The maximum in θ' runs over the keys with A > 0 (the keys a
    causal row sees)."""
    Ah = masked_weights(A, keep)
    o = A @ vproj
    oh = Ah @ vproj
    actual = np.abs(o - oh).sum(axis=1)
    nu = np.abs(vproj).sum(axis=1)                       # ||v'_i||_1
    a = (A * keep[None, :]).sum(axis=1)
    C = A @ nu
    P = (A * keep[None, :]) @ nu
    theta = C - (2.0 - 1.0 / a) * P
    numax = np.array([nu[A[r] > 0].max() for r in range(A.shape[0])])
    relaxed = 2.0 * (1.0 - a) * numax
    return actual, theta, relaxed


def perturbation_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, w_o: np.ndarray, h: int, group: int,
                      keep: np.ndarray, scale: Optional[float] = None, causal: bool = True):
    """(actual, θ, θ') as [G][W] arrays for the window rows of KV head h.

    q [G][W][d], k, v [n][d] float64; w_o [D][H*G*d] float64 (nn.Linear weight: query head
    h*G+g owns columns [(h*G+g)*d, +d)); keep: bool [n], the kept set of KV head h."""
    G, W, d = q.shape
    A = attention_rows(q, k, scale, causal)              # [G][W][n]
    out = np.zeros((3, G, W))
    for g in range(group):
        qh = h * group + g
        vproj = v @ w_o[:, qh * d:(qh + 1) * d].T        # [n][D]
        out[:, g, :] = perturbation_rows(A[g], vproj, keep)
    return out


def run_perturbation_layer(q_bits, k_bits, v_bits, w_o_bits, kept, *, group: int, scale=None,
                           causal: bool = True, heads=None):
    """Per request: float64 [H][3][G][W] (actual, θ, θ') for the kept sets kept[b][h]
    (position arrays)."""
    w_o = bf16_to_f64(w_o_bits)
    out = []
    for b in range(len(k_bits)):
        k = bf16_to_f64(k_bits[b])
        v = bf16_to_f64(v_bits[b])
        H, n, d = k.shape
        hs = range(H) if heads is None else heads
        r = np.full((H, 3, group, q_bits.shape[3]), np.nan)
        for h in hs:
            keep = np.zeros(n, bool)
            keep[np.asarray(kept[b][h], np.int64)] = True
            r[h] = perturbation_head(bf16_to_f64(q_bits[b][h]), k[h], v[h], w_o, h, group, keep, scale, causal)
        out.append(r)
    return out
