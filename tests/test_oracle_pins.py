"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Each test ties one oracle function to a hand-computed fixture (tests/golden), a closed
form, a library routine for a special case, brute force on tiny inputs, or an invariant
stated by the pages.  Together they are chosen so that a plausible slip (missing scale,
off-by-one causal mask, wrong reduction axis, transposed W_O, wrong pooling padding,
tie order) breaks at least one of them; test_oracle_mutants.py plants such slips.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.ndimage
import scipy.special

from oracle import kvsel_oracle as O
from kv_cache_eviction_window_gb300 import datagen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, rest = line.split(":", 1)
        vals[key.strip()] = [Fraction(t) for t in rest.split()]
    return vals


def f64(x):
    return np.array([float(v) for v in x])


# --------------------------------------------------------------------- decoding
def test_bf16_decode_closed_form():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F7F, 0x8000], np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 2.0 ** -133, (2 - 2.0 ** -7) * 2.0 ** 127, -0.0]
    got = O.bf16_to_f64(bits)
    assert list(got) == want


# --------------------------------------------------------------------- hand example
def hand_inputs():
    q = np.array([[[1.0, 0.0], [1.0, 0.0]]])            # [G=1][W=2][d=2]
    k = np.array([[i, 0.0] for i in range(4)])           # [n=4][d=2]
    return q, k, math.log(2.0)


def test_hand_softmax_rows():
    g = load_golden("hand_example.txt")
    q, k, sc = hand_inputs()
    p = O.softmax_rows(O.window_logits(q, k, sc, causal=True))
    np.testing.assert_allclose(p[0, 0], f64(g["p_row0"]), rtol=1e-14, atol=0)
    np.testing.assert_allclose(p[0, 1], f64(g["p_row1"]), rtol=1e-14, atol=0)
    assert p[0, 0, 3] == 0.0


@pytest.mark.parametrize("op,key", [("sum", "s_sum"), ("mean", "s_mean"), ("max", "s_max")])
def test_hand_reductions(op, key):
    g = load_golden("hand_example.txt")
    q, k, sc = hand_inputs()
    s = O.window_scores(q, k, op, sc, causal=True)
    np.testing.assert_allclose(s, f64(g[key]), rtol=1e-14)


def test_hand_pooling_and_selection():
    g = load_golden("hand_example.txt")
    s = f64(g["s_sum"])
    np.testing.assert_allclose(O.pool1d(s, "max", 3), f64(g["maxpool3_sum"]), rtol=1e-14)
    np.testing.assert_allclose(O.pool1d(s, "avg", 3), f64(g["avgpool3_sum"]), rtol=1e-14)
    none = np.zeros(4, bool)
    assert list(O.top_b(s, 2, none)) == [int(v) for v in g["top2_sum"]]
    assert list(O.top_b(O.pool1d(s, "max", 3), 2, none)) == [int(v) for v in g["top2_maxpool3"]]


def test_hand_value_norm_and_two_stage():
    g = load_golden("hand_example.txt")
    w_o = np.array([[1.0, 2.0], [3.0, -4.0]])
    v = np.array([[1.0, 1.0], [2.0, -1.0], [0.0, 0.0], [-1.0, 0.0]])
    nu = O.value_norm(v, w_o, h=0, group=1)
    np.testing.assert_array_equal(nu, f64(g["nu"]))
    s = f64(g["s_sum"])
    sv = O.combine(s, nu, 1e-4)
    np.testing.assert_allclose(sv, f64(g["s_val_sum"]), rtol=1e-14)
    none = np.zeros(4, bool)
    assert list(O.top_b(sv, 2, none)) == [int(x) for x in g["top2_val"]]
    assert list(O.select_two_stage(s, sv, 2, none, 0.5)) == [int(x) for x in g["two_stage_b2"]]


# --------------------------------------------------------------------- scoring
def test_textbook_softmax_special_case():
    """G = W = 1, no mask, no pooling: the score is the plain softmax of q K^T / sqrt(d)."""
    rng = np.random.default_rng(0)
    d, n = 16, 37
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((n, d))
    s = O.window_scores(q, k, "sum", None, causal=False)
    ref = scipy.special.softmax(k @ q[0, 0] / math.sqrt(d))
    np.testing.assert_allclose(s, ref, rtol=1e-13)
    s_mean = O.window_scores(q, k, "mean", None, causal=False)
    np.testing.assert_allclose(s_mean, ref, rtol=1e-13)


def test_causal_mask_positions_and_row_sums():
    rng = np.random.default_rng(1)
    G, W, d, n = 3, 5, 8, 11
    q = rng.standard_normal((G, W, d))
    k = rng.standard_normal((n, d))
    p = O.softmax_rows(O.window_logits(q, k, None, causal=True))
    for w in range(W):
        pos = n - W + w
        assert np.all(p[:, w, pos + 1:] == 0.0)
        assert np.all(p[:, w, :pos + 1] > 0.0)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-14)


def test_reductions_relate():
    rng = np.random.default_rng(2)
    G, W, d, n = 4, 6, 8, 20
    q = rng.standard_normal((G, W, d))
    k = rng.standard_normal((n, d))
    s_sum = O.window_scores(q, k, "sum")
    s_mean = O.window_scores(q, k, "mean")
    s_max = O.window_scores(q, k, "max")
    np.testing.assert_allclose(s_mean * G * W, s_sum, rtol=1e-13)
    # brute force over rows
    p = O.softmax_rows(O.window_logits(q, k, None, True))
    for i in range(n):
        assert s_max[i] == max(p[g, w, i] for g in range(G) for w in range(W))
    # the window rows are probability distributions: scores sum to the row count
    assert abs(s_sum.sum() - G * W) < 1e-12


def test_scale_enters_logits():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 2, 4))
    k = rng.standard_normal((6, 4))
    l1 = O.window_logits(q, k, None, causal=False)
    l2 = O.window_logits(q, k, 1.0, causal=False)
    np.testing.assert_allclose(l1 * 2.0, l2, rtol=1e-14)  # 1/sqrt(4) = 1/2


# --------------------------------------------------------------------- pooling
def test_pool_identity_and_global_max():
    rng = np.random.default_rng(4)
    s = rng.random(13)
    np.testing.assert_array_equal(O.pool1d(s, "max", 1), s)
    np.testing.assert_array_equal(O.pool1d(s, "avg", 1), s)
    np.testing.assert_array_equal(O.pool1d(s, "none", 7), s)
    np.testing.assert_array_equal(O.pool1d(s, "max", 2 * 13 - 1), np.full(13, s.max()))


@pytest.mark.parametrize("k", [3, 5, 7])
def test_pool_matches_library(k):
    rng = np.random.default_rng(5 + k)
    s = rng.random(50)
    ref_max = scipy.ndimage.maximum_filter1d(s, size=k, mode="nearest")
    np.testing.assert_array_equal(O.pool1d(s, "max", k), ref_max)
    ref_avg = np.convolve(s, np.ones(k), mode="same") / k
    np.testing.assert_allclose(O.pool1d(s, "avg", k), ref_avg, rtol=1e-14)


# --------------------------------------------------------------------- value norm
def test_value_norm_identity_slices_closed_form():
    """W_O^(h,g) = [I_d; 0] for every g: group sum gives G*||v||_1, per head the same."""
    rng = np.random.default_rng(6)
    H, G, d, D, n = 2, 3, 4, 6, 9
    w_o = np.zeros((D, H * G * d))
    for q in range(H * G):
        w_o[:d, q * d:(q + 1) * d] = np.eye(d)
    v = rng.standard_normal((n, d))
    for h in range(H):
        np.testing.assert_allclose(O.value_norm(v, w_o, h, G), G * np.abs(v).sum(1), rtol=1e-14)
        np.testing.assert_allclose(O.value_norm(v, w_o, h, G, "per_head"),
                                   G * np.abs(v).sum(1), rtol=1e-14)


def test_value_norm_l2_closed_forms():
    """L2 reading: identity slices give G*||v||_2; an orthogonal group sum Q (Q^T Q = I)
    preserves the Euclidean norm; one 3-4-5 row by hand."""
    rng = np.random.default_rng(23)
    H, G, d, D, n = 2, 3, 4, 6, 9
    w_o = np.zeros((D, H * G * d))
    for q in range(H * G):
        w_o[:d, q * d:(q + 1) * d] = np.eye(d)
    v = rng.standard_normal((n, d))
    for h in range(H):
        np.testing.assert_allclose(O.value_norm(v, w_o, h, G, norm="l2"), G * np.sqrt((v * v).sum(1)), rtol=1e-14)
    # orthogonal W_h (one query head per KV head): ||Q v||_2 = ||v||_2
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    w1 = np.zeros((d, d))
    w1[:, :] = Q
    np.testing.assert_allclose(O.value_norm(v, w1, 0, 1, norm="l2"), np.linalg.norm(v, axis=1), rtol=1e-13)
    # hand: W_h = diag(1, 1), v = (3, 4) -> 5 (L1 would give 7)
    w2 = np.eye(2)
    vv = np.array([[3.0, 4.0]])
    assert O.value_norm(vv, w2, 0, 1, norm="l2")[0] == 5.0
    assert O.value_norm(vv, w2, 0, 1, norm="l1")[0] == 7.0


def test_value_norm_l2_brute_force():
    rng = np.random.default_rng(24)
    H, G, d, D, n = 2, 2, 3, 5, 4
    w_o = rng.standard_normal((D, H * G * d))
    v = rng.standard_normal((n, d))
    for h in range(H):
        got = O.value_norm(v, w_o, h, G, norm="l2")
        for i in range(n):
            tot = 0.0
            for j in range(D):
                x = 0.0
                for g in range(G):
                    for c in range(d):
                        x += w_o[j, (h * G + g) * d + c] * v[i, c]
                tot += x * x
            assert abs(got[i] - math.sqrt(tot)) < 1e-12 * max(1.0, math.sqrt(tot))


def test_value_norm_readings_differ_on_opposite_slices():
    d, D, G = 3, 3, 2
    w_o = np.concatenate([np.eye(d), -np.eye(d)], axis=1)   # head 0: +I, head 1: -I
    v = np.array([[1.0, -2.0, 3.0]])
    assert O.value_norm(v, w_o, 0, G)[0] == 0.0
    assert O.value_norm(v, w_o, 0, G, "per_head")[0] == 12.0


def test_value_norm_brute_force():
    """Explicit loops over outputs j, columns c and group heads g on tiny random data."""
    rng = np.random.default_rng(7)
    H, G, d, D, n = 2, 2, 3, 5, 4
    w_o = rng.standard_normal((D, H * G * d))
    v = rng.standard_normal((n, d))
    for h in range(H):
        got = O.value_norm(v, w_o, h, G)
        got_i = O.value_norm(v, w_o, h, G, "per_head")
        for i in range(n):
            tot = 0.0
            tot_i = 0.0
            for j in range(D):
                acc = 0.0
                for g in range(G):
                    acc_g = 0.0
                    for c in range(d):
                        acc_g += w_o[j, (h * G + g) * d + c] * v[i, c]
                    acc += acc_g
                    tot_i += abs(acc_g)
                tot += abs(acc)
            assert abs(got[i] - tot) < 1e-12
            assert abs(got_i[i] - tot_i) < 1e-12


def test_value_norm_row_blocks_do_not_matter():
    rng = np.random.default_rng(8)
    w_o = rng.standard_normal((7, 2 * 2 * 4))
    v = rng.standard_normal((23, 4))
    a = O.value_norm(v, w_o, 1, 2, row_block=5)
    b = O.value_norm(v, w_o, 1, 2, row_block=4096)
    np.testing.assert_array_equal(a, b)


# --------------------------------------------------------------------- selection
def brute_top(scores, budget, forced):
    """Best subset by enumeration: contains every forced entry; compare subsets by their
    scores sorted descending, then by their indices sorted ascending."""
    n = len(scores)
    best = None
    for sub in itertools.combinations(range(n), budget):
        if not all(i in sub for i in np.flatnonzero(forced)):
            continue
        free = [i for i in sub if not forced[i]]
        key = (sorted((-scores[i] for i in free)), sorted(free))
        if best is None or key < best[0]:
            best = (key, sub)
    return list(best[1])


@pytest.mark.parametrize("seed", range(6))
def test_top_b_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(6, 12))
    s = rng.integers(0, 5, size=n).astype(float)   # many exact ties
    forced = np.zeros(n, bool)
    forced[rng.choice(n, size=int(rng.integers(0, 3)), replace=False)] = True
    for budget in range(int(forced.sum()), n + 1):
        assert list(O.top_b(s, budget, forced)) == brute_top(s, budget, forced)


def test_two_stage_degenerates_to_attention_only():
    """CriticalKV App. C.4 (Theorem C.1): with stage 2 scored like stage 1 the algorithm is
    the attention-only selection; alpha = 1 leaves no stage-2 budget."""
    rng = np.random.default_rng(9)
    n = 200
    s = rng.random(n)
    sv = rng.random(n)
    f = O.forced_mask(n, 4, 8)
    for b in (12, 50, 199):
        ref = O.top_b(s, b, f)
        np.testing.assert_array_equal(O.select_two_stage(s, s, b, f, 0.5), ref)
        np.testing.assert_array_equal(O.select_two_stage(s, sv, b, f, 1.0), ref)


def test_large_eps_ranks_by_value_norm():
    rng = np.random.default_rng(10)
    n = 64
    s = rng.random(n) * 1e-3
    nu = rng.random(n) + 0.5
    f = np.zeros(n, bool)
    sv = O.combine(s, nu, eps=1e6)
    np.testing.assert_array_equal(O.select_two_stage(s, sv, 20, f, 0.0), O.top_b(nu, 20, f))


def test_two_stage_brute_force():
    rng = np.random.default_rng(11)
    n = 10
    for _ in range(20):
        s = rng.integers(0, 4, n).astype(float)
        sv = rng.integers(0, 4, n).astype(float)
        f = np.zeros(n, bool)
        f[0] = True
        for b in range(1, n + 1):
            b1 = max(int(math.floor(0.5 * b)), 1)
            s1 = brute_top(s, b1, f)
            keep = np.zeros(n, bool)
            keep[s1] = True
            want = brute_top(sv, b, keep)
            assert list(O.select_two_stage(s, sv, b, f, 0.5)) == want


def test_selection_invariants_and_identity():
    rng = np.random.default_rng(12)
    n = 500
    s = rng.random(n)
    f = O.forced_mask(n, 4, 32)
    for b in (36, 100, 499, 500):
        idx = O.top_b(s, b, f)
        assert len(idx) == b
        assert np.all(np.diff(idx) > 0) and idx[0] >= 0 and idx[-1] < n
        assert set(np.flatnonzero(f)) <= set(idx.tolist())
    np.testing.assert_array_equal(O.top_b(s, n, f), np.arange(n))
    with pytest.raises(ValueError):
        O.top_b(s, 35, f)


def test_forced_mask():
    f = O.forced_mask(10, 4, 3)
    assert f.tolist() == [True] * 4 + [False] * 3 + [True] * 3
    assert O.forced_mask(5, 4, 0).tolist() == [True] * 4 + [False]


def test_per_layer_special_cases():
    rng = np.random.default_rng(13)
    H, n = 3, 40
    s = rng.random((H, n))
    none = np.zeros((H, n), bool)
    # no floor, no forced: plain flattened top-B
    got = O.select_per_layer(s, 30, none, 0)
    flat = np.sort(np.argsort(-s.reshape(-1), kind="stable")[:30])
    want = [flat[(flat >= h * n) & (flat < (h + 1) * n)] - h * n for h in range(H)]
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b)
    # one head: same as the per-head selection
    f = O.forced_mask(n, 4, 5)[None]
    np.testing.assert_array_equal(O.select_per_layer(s[:1], 17, f, 10)[0], O.top_b(s[0], 17, f[0]))


def test_per_layer_floors_invariants():
    rng = np.random.default_rng(14)
    H, n = 4, 300
    s = rng.random((H, n)) ** 4
    s[0] *= 10.0  # head 0 dominates the flattened order
    f = np.stack([O.forced_mask(n, 4, 16)] * H)
    budget, fl = 240, 30
    idx = O.select_per_layer(s, budget, f, fl)
    assert sum(len(i) for i in idx) == budget
    for h in range(H):
        assert len(idx[h]) >= fl
        assert set(np.flatnonzero(f[h])) <= set(idx[h].tolist())
        assert np.all(np.diff(idx[h]) > 0)
        # each head's floor picks are its own top entries
        assert set(O.top_b(s[h], fl, f[h]).tolist()) <= set(idx[h].tolist())
    # everything kept beyond the floors outranks everything dropped
    kept = np.zeros((H, n), bool)
    for h in range(H):
        kept[h, idx[h]] = True
    floor_keep = np.zeros((H, n), bool)
    for h in range(H):
        floor_keep[h, O.top_b(s[h], fl, f[h])] = True
    extra = kept & ~floor_keep
    dropped = ~kept
    assert s[extra].min() >= s[dropped].max()


# --------------------------------------------------------------------- permutation
def test_permutation_consistency():
    """Permuting prefix keys that every window row sees permutes the scores (no pooling)."""
    rng = np.random.default_rng(15)
    G, W, d, n = 2, 4, 8, 40
    q = rng.standard_normal((G, W, d))
    k = rng.standard_normal((n, d))
    lo, hi = 4, n - W
    perm = np.arange(n)
    perm[lo:hi] = lo + rng.permutation(hi - lo)
    s = O.window_scores(q, k, "mean")
    sp = O.window_scores(q, k[perm], "mean")
    np.testing.assert_allclose(sp, s[perm], rtol=1e-12)
    f = O.forced_mask(n, 4, W)
    a = O.top_b(s, 15, f)
    b = O.top_b(sp, 15, f)
    np.testing.assert_array_equal(np.sort(perm[b]), a)


# --------------------------------------------------------------------- query-agnostic
def test_query_agnostic_brute_force_and_chunks():
    rng = np.random.default_rng(16)
    G, m, d, n = 2, 7, 4, 9
    q = rng.standard_normal((G, m, d))
    k = rng.standard_normal((n, d))
    S = O.query_agnostic_scores(q, k)
    for i in range(n):
        best = 0.0
        for g in range(G):
            for j in range(m):
                logits = [float(q[g, j] @ k[t]) / math.sqrt(d) for t in range(n)]
                mx = max(logits)
                z = sum(math.exp(x - mx) for x in logits)
                best = max(best, math.exp(logits[i] - mx) / z)
        assert abs(S[i] - best) < 1e-14
    np.testing.assert_array_equal(O.query_agnostic_scores(q, k, q_chunk=3), S)


def test_max_trick_identity():
    """max_r softmax_r[i] == exp(max_r (l_ri - logsumexp_r)) on small inputs."""
    rng = np.random.default_rng(17)
    q = rng.standard_normal((1, 64, 8))
    k = rng.standard_normal((64, 8))
    l = (q[0] @ k.T) / math.sqrt(8)
    c = scipy.special.logsumexp(l, axis=1)
    np.testing.assert_allclose(np.exp((l - c[:, None]).max(axis=0)),
                               O.query_agnostic_scores(q, k), rtol=1e-13)


def test_logit_score_brute_force_and_chunks():
    """KVzip-logit: max over group heads and positions of the scaled dot product, by
    plain loops; chunking does not change it."""
    rng = np.random.default_rng(21)
    G, m, d, n = 3, 5, 4, 8
    q = rng.standard_normal((G, m, d))
    k = rng.standard_normal((n, d))
    S = O.query_agnostic_logit_scores(q, k)
    for i in range(n):
        best = -math.inf
        for g in range(G):
            for j in range(m):
                best = max(best, sum(float(q[g, j, c]) * float(k[i, c]) for c in range(d)) / math.sqrt(d))
        assert abs(S[i] - best) < 1e-14
    np.testing.assert_array_equal(O.query_agnostic_logit_scores(q, k, q_chunk=2), S)
    np.testing.assert_allclose(O.query_agnostic_logit_scores(q, k, scale=0.5), S * math.sqrt(d) * 0.5, rtol=1e-14)


def test_logit_and_softmax_scores_rank_alike_for_one_query():
    """With a single query row the softmax weight is exp(logit - logsumexp): a monotone
    function of the logit, so the two scores order the keys identically."""
    rng = np.random.default_rng(22)
    q = rng.standard_normal((1, 1, 16))
    k = rng.standard_normal((40, 16))
    sl = O.query_agnostic_logit_scores(q, k)
    ss = O.query_agnostic_scores(q, k)
    np.testing.assert_allclose(ss, np.exp(sl - scipy.special.logsumexp(sl)), rtol=1e-13)
    np.testing.assert_array_equal(np.argsort(-sl, kind="stable"), np.argsort(-ss, kind="stable"))


def test_head_scores():
    S = np.array([[1.0, 5.0, 3.0], [-2.0, -1.0, -7.0], [0.25, 0.25, 0.5]])
    np.testing.assert_array_equal(O.head_scores(S), [5.0, -1.0, 0.5])
    # a head whose keys all score the same has that score as its head score
    assert O.head_scores(np.full((1, 9), 0.125))[0] == 0.125


# --------------------------------------------------------------------- compaction
def test_compact_and_paging():
    wl = datagen.WORKLOADS[4].replace(batch=3, n_min=40, n_ctx=90)
    inp = datagen.make_layer(wl, 0)
    pg = inp["paged"]
    for b, n in enumerate(inp["n_ctx"]):
        kb = O.unpage(pg["k_pool"], pg["block_table"][b], n)
        vb = O.unpage(pg["v_pool"], pg["block_table"][b], n)
        np.testing.assert_array_equal(kb, inp["k"][b])
        np.testing.assert_array_equal(vb, inp["v"][b])
    k = inp["k"][0][0]
    idx = np.array([0, 3, 17, 39])
    np.testing.assert_array_equal(O.compact(k, idx), np.stack([k[i] for i in idx]))
    np.testing.assert_array_equal(O.compact(k, np.arange(k.shape[0])), k)


def test_two_stage_per_layer_budget_hand_example():
    """CriticalKV Algorithm 2 line 1 then Algorithm 1 per head, by hand: two heads of four
    entries, layer budget 4, no forced entries, no floor, alpha = 0.5.  The pooled scores
    put three of the layer's top four in head 0 and one in head 1, so b_0 = 3, b_1 = 1.
    Head 0: stage 1 keeps floor(1.5) = 1 entry by score (entry 0), stage 2 the two best
    of the others by s_val (entries 2 and 3, s_val 9 and 5; entry 2 has the lowest pooled
    score of the head).  Head 1: stage 1 keeps floor(0.5) = 0, so
    stage 2 takes the single best s_val (entry 2), though its pooled score is lowest."""
    s_pool = np.array([[0.9, 0.8, 0.1, 0.7], [0.6, 0.05, 0.01, 0.02]])
    s_val = np.array([[1.0, 2.0, 9.0, 5.0], [0.1, 0.2, 7.0, 0.3]])
    fm = np.zeros((2, 4), dtype=bool)
    out = O.select_two_stage_per_layer(s_pool, s_val, 4, fm, 0, 0.5)
    assert out[0].tolist() == [0, 2, 3]
    assert out[1].tolist() == [2]


@pytest.mark.parametrize("seed", range(4))
def test_two_stage_per_layer_budget_invariants(seed):
    """Per head: the allocation of the layer budget (counts add up to B_L, each at least
    the floor), two-stage selection within it (alpha = 1 gives back the attention-only
    per-layer selection), forced entries always kept."""
    rng = np.random.default_rng(seed)
    H, n = 3, 40
    s_pool = rng.random((H, n))
    s_val = rng.random((H, n))
    fm = np.stack([O.forced_mask(n, 2, 3)] * H)
    B_L, fl = 45, 8
    out = O.select_two_stage_per_layer(s_pool, s_val, B_L, fm, fl, 0.5)
    alloc = O.select_per_layer(s_pool, B_L, fm, fl)
    assert [len(x) for x in out] == [len(x) for x in alloc]
    assert sum(len(x) for x in out) == B_L and all(len(x) >= fl for x in out)
    for h in range(H):
        assert set(np.flatnonzero(fm[h]).tolist()) <= set(out[h].tolist())
        np.testing.assert_array_equal(out[h], O.select_two_stage(s_pool[h], s_val[h], len(alloc[h]), fm[h], 0.5))
    same = O.select_two_stage_per_layer(s_pool, s_val, B_L, fm, fl, 1.0)
    for h in range(H):
        np.testing.assert_array_equal(same[h], alloc[h])


# --------------------------------------------------------------------- partition / archive
def test_partition_hand_example():
    """VestigeKV §4.1: eviction archives rows instead of deleting them.  By hand: of the
    positions 0..5, keeping 0, 2 and 5 leaves 1, 3 and 4 for the archive; the archived
    rows are those rows in position order."""
    kept, ev = O.partition(6, np.array([5, 0, 2]))
    assert kept.tolist() == [0, 2, 5]
    assert ev.tolist() == [1, 3, 4]
    x = np.arange(12, dtype=np.uint16).reshape(6, 2)
    np.testing.assert_array_equal(O.archive(x, np.array([0, 2, 5])), np.array([[2, 3], [6, 7], [8, 9]]))


@pytest.mark.parametrize("seed", range(6))
def test_partition_invariants_and_reassembly(seed):
    """Both sides ascending, disjoint, together exactly [0, n); kept rows and archived rows
    put back at their positions give the cache again, bit for bit."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 300))
    b = int(rng.integers(0, n + 1))
    idx = np.sort(rng.choice(n, size=b, replace=False))
    kept, ev = O.partition(n, idx)
    assert np.all(np.diff(kept) > 0) and np.all(np.diff(ev) > 0)
    assert len(kept) + len(ev) == n
    assert not set(kept.tolist()) & set(ev.tolist())
    assert sorted(kept.tolist() + ev.tolist()) == list(range(n))
    x = rng.integers(0, 1 << 16, size=(n, 4), dtype=np.uint16)
    back = np.zeros_like(x)
    back[kept] = O.compact(x, idx)
    back[ev] = O.archive(x, idx)
    np.testing.assert_array_equal(back, x)


def test_partition_extremes():
    kept, ev = O.partition(5, np.arange(5))
    assert kept.tolist() == list(range(5)) and ev.size == 0
    kept, ev = O.partition(5, np.array([], dtype=np.int64))
    assert kept.size == 0 and ev.tolist() == list(range(5))
    assert O.archive(np.zeros((0, 3)), np.array([], dtype=np.int64)).shape == (0, 3)


# --------------------------------------------------------------------- end to end
def test_run_layer_small_invariants():
    wl = datagen.WORKLOADS[2].replace(layers=1, n_ctx=700, d_model=256)
    inp = datagen.make_layer(wl, 0, n_ctx=700)
    r = O.run_workload_layer(wl, inp)[0]
    B = O.head_budget(700, wl.budget_ratio)
    f = O.forced_mask(700, 4, 32)
    for h in range(wl.h_kv):
        assert len(r["idx"][h]) == B
        assert set(np.flatnonzero(f)) <= set(r["idx"][h].tolist())
        np.testing.assert_array_equal(r["k_out"][h], inp["k"][0][h][r["idx"][h]])
    assert np.all(r["nu"] > 0)
    np.testing.assert_allclose(r["s_raw"].sum(1), 1.0 * 1, rtol=1e-9)  # mean of prob rows


# --------------------------------------------------------------------- AnchorKV anchors
from oracle import anchor_oracle as A  # noqa: E402


def test_anchor_count_closed_form():
    # AnchorKV §4.1: k = S/128; the recent window counts inside k (§3.2); never above n
    assert A.anchor_count(32768, 32) == 256
    assert A.anchor_count(131072, 64) == 1024
    assert A.anchor_count(1000, 32) == 32       # floor(1000/128) = 7 < |F|
    assert A.anchor_count(20, 20) == 20
    assert A.anchor_count(0, 0) == 0


def test_select_anchors_hand_example():
    # n = 12, recent window {10, 11}, k = 7, rho = 0.7: stage 1 = F + floor(0.7 * 5) = 3
    # picks by score among 0..9: 0.9 (5), then the tie 0.5 at 1 and 3 (index order);
    # stage 2 = 2 picks by random key among the rest: the 0.99 at 1 is taken already, so
    # the three-way tie 0.7 at {2, 4, 8} resolves to 2 and 4.
    s = np.array([0.1, 0.5, 0.3, 0.5, 0.2, 0.9, 0.0, 0.3, 0.4, 0.1, 0.05, 0.01])
    r = np.array([0.2, 0.99, 0.7, 0.1, 0.7, 0.3, 0.6, 0.05, 0.7, 0.4, 0.8, 0.9])
    fm = O.forced_mask(12, 0, 2)
    got = A.select_anchors(s, r, 7, fm, 0.7)
    assert got.tolist() == [1, 2, 3, 4, 5, 10, 11]


def test_select_anchors_rho_extremes():
    g = np.random.default_rng(5)
    n, k = 300, 40
    s = g.random(n)
    r = g.random(n)
    fm = O.forced_mask(n, 0, 16)
    # rho = 1: all free slots by score = the plain top-k with the window forced
    assert np.array_equal(A.select_anchors(s, r, k, fm, 1.0), O.top_b(s, k, fm))
    # rho = 0: all free slots by the random keys
    assert np.array_equal(A.select_anchors(s, r, k, fm, 0.0), O.top_b(r, k, fm))


def test_select_anchors_random_share_is_uniform_without_replacement():
    # n = 40, F = 4 recent, k = 12, rho = 0.5: 4 by score, then 4 drawn from the other 32
    g = np.random.default_rng(11)
    n, k, trials = 40, 12, 3000
    s = np.linspace(1.0, 0.0, n)          # stage 1 is always positions 0..3
    fm = O.forced_mask(n, 0, 4)
    counts = np.zeros(n, int)
    for _ in range(trials):
        got = A.select_anchors(s, g.random(n), k, fm, 0.5)
        assert len(got) == k and len(set(got.tolist())) == k
        counts[got] += 1
    assert (counts[:4] == trials).all() and (counts[-4:] == trials).all()
    mid = counts[4:n - 4]                 # 32 positions, 4 draws each trial: 375 expected
    assert abs(mid.sum() - 4 * trials) == 0
    assert mid.min() > 375 - 100 and mid.max() < 375 + 100


def test_anchor_project_scaled_basis():
    # anchors c_j e_j: cos(x, a_j) = x_j / |x|, so the slot is the largest coordinate
    # (signed) and gamma = x_j / c_j
    c = [2.0, 0.5, 3.0, 1.0]
    x = np.zeros((6, 4))
    for j in range(4):
        x[j, j] = c[j]
    x[4] = [1.0, -2.0, 0.5, 0.7]
    x[5] = [-1.0, -2.0, -0.5, -3.0]
    slot, gamma, _ = A.anchor_project(x, np.arange(4))
    assert slot.tolist() == [0, 1, 2, 3, 0, 2]
    assert np.allclose(gamma, [1, 1, 1, 1, 0.5, -0.5 / 3.0], rtol=0, atol=1e-15)


def test_anchor_project_parallel_zero_and_duplicates():
    a = np.array([1.0, 2.0, -2.0])
    b = np.array([0.0, 1.0, 0.0])
    x = np.stack([a, a.copy(), b, 2.5 * b, np.zeros(3), -a, a])
    anchors = np.array([0, 1, 2])           # anchors 0 and 1 hold the same vector
    slot, gamma, cos = A.anchor_project(x, anchors)
    assert slot[:3].tolist() == [0, 1, 2] and (gamma[:3] == 1.0).all()   # anchors: themselves
    assert slot[3] == 2 and gamma[3] == 2.5                              # parallel to b
    assert slot[4] == 0 and gamma[4] == 0.0                              # zero vector: slot 0
    # -a: cos -1 with anchors 0, 1 and -2/3 with b: the larger (signed) cosine is b's
    assert slot[5] == 2 and abs(gamma[5] - (-2.0)) < 1e-15
    assert slot[6] == 0 and gamma[6] == 1.0                              # tie: first slot


def test_anchor_project_residual_orthogonal_and_best():
    g = np.random.default_rng(3)
    x = g.standard_normal((200, 16))
    anchors = np.sort(g.choice(200, 12, replace=False))
    slot, gamma, cos = A.anchor_project(x, anchors)
    a = x[anchors][slot]
    r = x - gamma[:, None] * a
    # the residual of an orthogonal projection is orthogonal to the anchor
    assert np.abs((r * a).sum(1)).max() < 1e-12 * np.abs(x).max() ** 2 * 16
    # and no other anchor has a larger cosine
    assert (cos[np.arange(200), slot] >= cos.max(1) - 1e-15).all()
    # |r|^2 = |x|^2 (1 - cos^2) for the chosen anchor (Pythagoras)
    xn2 = (x * x).sum(1)
    c = cos[np.arange(200), slot]
    nonanchor = np.setdiff1d(np.arange(200), anchors)
    assert np.allclose((r * r).sum(1)[nonanchor], (xn2 * (1 - c * c))[nonanchor], rtol=1e-9, atol=1e-12)


def test_run_anchor_layer_invariants():
    wl = datagen.WORKLOADS[6].replace(h_kv=2, n_ctx=700)
    inp = datagen.make_layer(wl, 0, n_ctx=700)
    r = A.run_anchor_workload_layer(wl, inp)[0]
    assert r["k"] == 32                         # floor(700/128) = 5 < W = 32
    wl2 = wl.replace(n_ctx=9000)
    inp2 = datagen.make_layer(wl2, 0, n_ctx=9000)
    r2 = A.run_anchor_workload_layer(wl2, inp2, heads=[0])[0]
    assert r2["k"] == 70
    anc = r2["anchors"][0]
    assert len(anc) == 70 and np.all(np.diff(anc) > 0)
    assert set(range(9000 - 32, 9000)) <= set(anc.tolist())
    # 32 forced + floor(0.7 * 38) = 26 by score: all of them rank above the random ones
    s = r2["s_pool"][0]
    free = np.setdiff1d(anc, np.arange(9000 - 32, 9000))
    top26 = O.top_b(s, 58, O.forced_mask(9000, 0, 32))
    assert set(top26.tolist()) <= set(anc.tolist())
    assert len(free) == 38


# --------------------------------------------------------------------- output perturbation
from oracle import perturb_oracle as PO  # noqa: E402


def test_perturbation_two_keys_hand_example():
    # A = (3/4, 1/4), keep {0}: ô = v'_0, o - ô = 1/4 (v'_1 - v'_0) = (0.5, 0.75);
    # θ = A_1 (||v'_0|| + ||v'_1||) = 1/4 * 7; θ' = 2 * 1/4 * max(3, 4)
    A = np.array([[0.75, 0.25]])
    vp = np.array([[1.0, -2.0], [3.0, 1.0]])
    actual, theta, relaxed = PO.perturbation_rows(A, vp, np.array([True, False]))
    assert actual[0] == 1.25 and abs(theta[0] - 1.75) < 1e-15 and relaxed[0] == 2.0


def test_perturbation_keep_all_is_zero_and_mask_renormalises():
    g = np.random.default_rng(2)
    A = g.random((5, 9))
    A /= A.sum(1, keepdims=True)
    vp = g.standard_normal((9, 6))
    actual, theta, relaxed = PO.perturbation_rows(A, vp, np.ones(9, bool))
    assert np.abs(actual).max() < 1e-12 and np.abs(theta).max() < 1e-12 and np.abs(relaxed).max() < 1e-12
    keep = np.array([1, 0, 1, 1, 0, 0, 1, 0, 1], bool)
    Ah = PO.masked_weights(A, keep)
    assert np.allclose(Ah.sum(1), 1.0) and (Ah[:, ~keep] == 0).all()
    # kept weights scale by 1 / kept mass (CriticalKV Theorem 3.2)
    assert np.allclose(Ah[:, keep], A[:, keep] / (A[:, keep].sum(1, keepdims=True)))


def test_perturbation_bound_chain():
    # triangle inequality: actual <= θ <= θ' for any kept set
    g = np.random.default_rng(8)
    for _ in range(20):
        n = 12
        A = g.random((4, n)) ** 3
        A /= A.sum(1, keepdims=True)
        vp = g.standard_normal((n, 5)) * g.random((n, 1)) * 3
        keep = g.random(n) < 0.5
        keep[0] = True
        actual, theta, relaxed = PO.perturbation_rows(A, vp, keep)
        assert (actual <= theta + 1e-12).all() and (theta <= relaxed + 1e-12).all()


def test_relaxed_bound_minimised_by_attention_only_selection():
    # CriticalKV Theorem C.1: over all kept sets of size B, the top-B by A minimises θ'
    g = np.random.default_rng(4)
    n, B = 7, 3
    A = g.random((1, n))
    A /= A.sum()
    vp = g.standard_normal((n, 4))
    best = min(PO.perturbation_rows(A, vp, np.isin(np.arange(n), s))[2][0]
               for s in itertools.combinations(range(n), B))
    top = np.argsort(-A[0])[:B]
    got = PO.perturbation_rows(A, vp, np.isin(np.arange(n), top))[2][0]
    assert abs(got - best) < 1e-12


def test_perturbation_head_uses_its_own_w_o_slice():
    # only query head (h, g) = (1, 1) of H = 3, G = 2 has a non-zero slice [I_d; 0]: its
    # projected values are the raw values, every other query head sees zeros
    g = np.random.default_rng(6)
    H, G, d, D, n, W = 3, 2, 4, 6, 10, 3
    q = g.standard_normal((G, W, d))
    k = g.standard_normal((n, d))
    v = g.standard_normal((n, d))
    w_o = np.zeros((D, H * G * d))
    qh = 1 * G + 1
    w_o[:d, qh * d:(qh + 1) * d] = np.eye(d)
    keep = np.zeros(n, bool)
    keep[[0, 3, 7, 8, 9]] = True
    out = PO.perturbation_head(q, k, v, w_o, 1, G, keep)
    A = PO.attention_rows(q, k)
    want = np.abs((A[1] - PO.masked_weights(A[1], keep)) @ v).sum(1)
    assert np.allclose(out[0, 1], want, rtol=1e-12, atol=1e-14)
    assert np.abs(out[:, 0]).max() == 0.0


def test_relaxed_bound_runs_over_the_keys_a_row_sees():
    # the third key carries zero weight (a causal row does not see it): its large norm
    # must not enter θ' = 2 (1 - a) max ||v'_i||_1
    A = np.array([[0.5, 0.5, 0.0]])
    vp = np.array([[1.0, 0.0], [0.0, -2.0], [100.0, 0.0]])
    _, _, relaxed = PO.perturbation_rows(A, vp, np.array([True, False, False]))
    assert relaxed[0] == 2.0 * 0.5 * 2.0
