"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch them.

Each mutant replaces one oracle function with a subtly wrong version; the pin tests of
test_oracle_pins.py are then run against the mutated module and at least one must fail.
"""
import math

import numpy as np
import pytest

from oracle import kvsel_oracle as O
import tests.test_oracle_pins as P

from oracle import anchor_oracle as AO
from oracle import perturb_oracle as PO

ORIG = {name: getattr(O, name) for name in dir(O) if callable(getattr(O, name))}
A_ORIG = {name: getattr(AO, name) for name in dir(AO) if callable(getattr(AO, name))}
P_ORIG = {name: getattr(PO, name) for name in dir(PO) if callable(getattr(PO, name))}


def _logits_no_scale(q, k, scale=None, causal=True):
    return ORIG["window_logits"](q, k, 1.0, causal)


def _logits_causal_off_by_one(q, k, scale=None, causal=True):
    G, W, d = q.shape
    n = k.shape[0]
    if scale is None or scale == 0.0:
        scale = 1.0 / math.sqrt(d)
    l = np.matmul(q.reshape(G * W, d), k.T).reshape(G, W, n) * scale
    if causal:
        pos = n - W + np.arange(W)
        mask = np.arange(n)[None, :] >= pos[:, None]
        l = np.where(mask[None], -np.inf, l)
    return l


def _reduce_mean_over_group_only(p, op):
    if op == "mean":
        return p.sum(axis=1).mean(axis=0) if p.ndim == 3 else p.mean(axis=0)
    return ORIG["reduce_rows"](p, op)


def _avgpool_divides_by_count(s, kind, kernel):
    if kind != "avg" or kernel <= 1:
        return ORIG["pool1d"](s, kind, kernel)
    n = s.shape[0]
    h = kernel // 2
    out = np.empty(n)
    for i in range(n):
        a, b = max(0, i - h), min(n, i + h + 1)
        out[i] = s[a:b].mean()
    return out


def _value_norm_l2(v, w_o, h, group, mode="group_sum", row_block=4096, norm="l1"):
    sl = O.wo_slices(w_o, h, group, v.shape[1])
    wbar = sum(sl)
    return np.sqrt(((v @ wbar.T) ** 2).sum(1))


def _value_norm_first_slice_only(v, w_o, h, group, mode="group_sum", row_block=4096, norm="l1"):
    sl = O.wo_slices(w_o, h, group, v.shape[1])
    x = v @ (group * sl[0]).T
    return np.abs(x).sum(1) if norm == "l1" else np.sqrt((x * x).sum(1))


def _combine_no_eps(s_pool, nu, eps=1e-4):
    return s_pool * nu


def _top_b_ties_descending(scores, budget, forced):
    n = scores.shape[0]
    key = np.where(forced, np.inf, scores)
    order = np.lexsort((-np.arange(n), -key))
    return np.sort(order[:budget])


def _two_stage_ceil(s_pool, s_val, budget, forced, alpha=0.5):
    b1 = int(math.ceil(alpha * budget))
    s1 = ORIG["top_b"](s_pool, max(b1, int(forced.sum())), forced)
    keep = np.zeros_like(forced)
    keep[s1] = True
    return ORIG["top_b"](s_val, budget, keep)


def _two_stage_without_stage1(s_pool, s_val, budget, forced, alpha=0.5):
    return ORIG["top_b"](s_val, budget, forced)


def _forced_recent_off_by_one(n, n_sink, n_recent):
    f = np.zeros(n, dtype=bool)
    f[:n_sink] = True
    if n_recent > 0:
        f[max(n - n_recent - 1, 0):] = True
    return f


def _query_agnostic_mean(q, k, scale=None, q_chunk=0):
    G, m, d = q.shape
    p = O.softmax_rows((q.reshape(-1, d) @ k.T) / math.sqrt(d))
    return p.mean(axis=0)


def _per_layer_ignores_floor(scores, budget, forced, floor_per_head):
    return ORIG["select_per_layer"](scores, budget, forced, 0)


def _logit_no_scale(q, k, scale=None, q_chunk=0):
    return ORIG["query_agnostic_logit_scores"](q, k, 1.0, q_chunk)


def _logit_first_group_head_only(q, k, scale=None, q_chunk=0):
    return ORIG["query_agnostic_logit_scores"](q[:1], k, scale, q_chunk)


def _head_scores_mean(S):
    return S.mean(axis=1)


def _value_norm_l2_no_sqrt(v, w_o, h, group, mode="group_sum", row_block=4096, norm="l1"):
    r = ORIG["value_norm"](v, w_o, h, group, mode, row_block, norm)
    return r * r if norm == "l2" else r


def _anchor_abs_cosine(x, anchors):
    slot, gamma, cos = A_ORIG["anchor_project"](x, anchors)
    anchors = np.asarray(anchors, dtype=np.int64)
    A_ = x[anchors]
    an2 = (A_ * A_).sum(1)
    s2 = np.argmax(np.abs(cos), axis=1)
    g2 = (x @ A_.T)[np.arange(len(x)), s2] / np.where(an2[s2] > 0, an2[s2], 1.0)
    s2[anchors] = np.arange(len(anchors))
    g2[anchors] = 1.0
    return s2, g2, cos


def _anchor_gamma_unnormalised(x, anchors):
    slot, gamma, cos = A_ORIG["anchor_project"](x, anchors)
    an = np.sqrt((x[np.asarray(anchors, dtype=np.int64)] ** 2).sum(1))
    return slot, gamma * an[slot], cos


def _anchor_no_self(x, anchors):
    anchors = np.asarray(anchors, dtype=np.int64)
    slot, gamma, cos = A_ORIG["anchor_project"](x, anchors)
    best = np.argmax(cos, axis=1)
    slot[anchors] = best[anchors]
    return slot, gamma, cos


def _anchor_rho_ceil(s_pool, rand_key, k, forced, rho=0.7):
    nf = int(forced.sum())
    k1 = nf + int(math.ceil(rho * (k - nf)))
    s1 = O.top_b(s_pool, k1, forced)
    keep1 = np.zeros_like(forced)
    keep1[s1] = True
    return O.top_b(rand_key, k, keep1)


def _anchor_random_share_ignores_stage1(s_pool, rand_key, k, forced, rho=0.7):
    nf = int(forced.sum())
    k1 = nf + int(math.floor(rho * (k - nf)))
    s1 = O.top_b(s_pool, k1, forced)
    s2 = O.top_b(rand_key, k - k1 + nf, forced)
    return np.union1d(s1, s2)


def _anchor_count_ignores_forced(n, n_forced, div=128):
    return min(n, n // div)


def _pt_no_renormalise(A, keep):
    return A * keep[None, :]


def _pt_theta_2_minus_a(A, vproj, keep):
    actual, theta, relaxed = P_ORIG["perturbation_rows"](A, vproj, keep)
    nu = np.abs(vproj).sum(axis=1)
    a = (A * keep[None, :]).sum(axis=1)
    C = A @ nu
    P = (A * keep[None, :]) @ nu
    return actual, C - (2.0 - a) * P, relaxed


def _pt_relaxed_all_keys(A, vproj, keep):
    actual, theta, relaxed = P_ORIG["perturbation_rows"](A, vproj, keep)
    a = (A * keep[None, :]).sum(axis=1)
    return actual, theta, 2.0 * (1.0 - a) * np.abs(vproj).sum(axis=1).max()


def _pt_slice_transposed(q, k, v, w_o, h, group, keep, scale=None, causal=True):
    G, W, d = q.shape
    H = w_o.shape[1] // (group * d)
    A = PO.attention_rows(q, k, scale, causal)
    out = np.zeros((3, G, W))
    for g in range(group):
        qh = g * H + h                                    # query heads numbered g-major
        vproj = v @ w_o[:, qh * d:(qh + 1) * d].T
        out[:, g, :] = PO.perturbation_rows(A[g], vproj, keep)
    return out


def _two_stage_per_layer_uniform_split(s_pool, s_val, budget, forced, floor_per_head, alpha=0.5):
    H = s_pool.shape[0]
    b = budget // H
    return [O.select_two_stage(s_pool[h], s_val[h], b, forced[h], alpha) for h in range(H)]


def _partition_drops_last(n, idx):
    kept = np.zeros(n, dtype=bool)
    kept[np.asarray(idx, dtype=np.int64)] = True
    return np.flatnonzero(kept), np.flatnonzero(~kept[:-1])


def _partition_one_based(n, idx):
    kept = np.zeros(n + 1, dtype=bool)
    kept[np.asarray(idx, dtype=np.int64) + 1] = True
    return np.flatnonzero(kept[:n]), np.flatnonzero(~kept[:n])


def _archive_descending(x, idx):
    return x[O.partition(x.shape[0], idx)[1][::-1]]


P_MUTANTS = {
    "perturbation_no_renormalise": ("masked_weights", _pt_no_renormalise),
    "perturbation_theta_2_minus_a": ("perturbation_rows", _pt_theta_2_minus_a),
    "perturbation_relaxed_all_keys": ("perturbation_rows", _pt_relaxed_all_keys),
    "perturbation_slice_g_major": ("perturbation_head", _pt_slice_transposed),
}


A_MUTANTS = {
    "anchor_abs_cosine": ("anchor_project", _anchor_abs_cosine),
    "anchor_gamma_unnormalised": ("anchor_project", _anchor_gamma_unnormalised),
    "anchor_no_self": ("anchor_project", _anchor_no_self),
    "anchor_rho_ceil": ("select_anchors", _anchor_rho_ceil),
    "anchor_random_share_ignores_stage1": ("select_anchors", _anchor_random_share_ignores_stage1),
    "anchor_count_ignores_forced": ("anchor_count", _anchor_count_ignores_forced),
}


MUTANTS = {
    "no_scale": ("window_logits", _logits_no_scale),
    "causal_off_by_one": ("window_logits", _logits_causal_off_by_one),
    "mean_over_group_only": ("reduce_rows", _reduce_mean_over_group_only),
    "avgpool_divides_by_count": ("pool1d", _avgpool_divides_by_count),
    "value_norm_l2": ("value_norm", _value_norm_l2),
    "value_norm_first_slice": ("value_norm", _value_norm_first_slice_only),
    "combine_no_eps": ("combine", _combine_no_eps),
    "ties_descending": ("top_b", _top_b_ties_descending),
    "two_stage_ceil": ("select_two_stage", _two_stage_ceil),
    "two_stage_skips_stage1": ("select_two_stage", _two_stage_without_stage1),
    "forced_recent_off_by_one": ("forced_mask", _forced_recent_off_by_one),
    "query_agnostic_mean": ("query_agnostic_scores", _query_agnostic_mean),
    "per_layer_ignores_floor": ("select_per_layer", _per_layer_ignores_floor),
    "logit_no_scale": ("query_agnostic_logit_scores", _logit_no_scale),
    "logit_first_group_head": ("query_agnostic_logit_scores", _logit_first_group_head_only),
    "head_scores_mean": ("head_scores", _head_scores_mean),
    "value_norm_l2_no_sqrt": ("value_norm", _value_norm_l2_no_sqrt),
    "partition_drops_last": ("partition", _partition_drops_last),
    "two_stage_per_layer_uniform_split": ("select_two_stage_per_layer", _two_stage_per_layer_uniform_split),
    "partition_one_based": ("partition", _partition_one_based),
    "archive_descending": ("archive", _archive_descending),
}


def _pin_calls():
    calls = []
    for name in dir(P):
        if not name.startswith("test_"):
            continue
        fn = getattr(P, name)
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if not params:
            calls.append((name, fn, {}))
            continue
        argnames, values = params[0].args[0], params[0].args[1]
        names = [a.strip() for a in argnames.split(",")]
        for val in values:
            vals = val if isinstance(val, tuple) else (val,)
            calls.append((f"{name}{vals}", fn, dict(zip(names, vals))))
    return calls


@pytest.mark.parametrize("mutant", sorted(MUTANTS) + sorted(A_MUTANTS) + sorted(P_MUTANTS))
def test_pins_catch_mutant(mutant, monkeypatch):
    if mutant in P_MUTANTS:
        attr, fake = P_MUTANTS[mutant]
        monkeypatch.setattr(PO, attr, fake)
    elif mutant in A_MUTANTS:
        attr, fake = A_MUTANTS[mutant]
        monkeypatch.setattr(AO, attr, fake)
    else:
        attr, fake = MUTANTS[mutant]
        monkeypatch.setattr(O, attr, fake)
    failed = []
    for name, fn, kw in _pin_calls():
        try:
            fn(**kw)
        except (Exception, pytest.fail.Exception):
            failed.append(name)
    assert failed, f"no pin caught mutant {mutant}"
