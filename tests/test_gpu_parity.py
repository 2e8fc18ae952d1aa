"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on seeded inputs.

Sizes span several key tiles and a ragged tail; full-size layers are checked on every
score where the oracle is cheap, and on sampled values plus size-independent properties
where it is not.  Tolerances (tests/gpu_harness.py): scores within 1e-3 relative (plus
an absolute floor of 1e-7 x the head's max for flushed denormals); kept sets equal
except entries within 1e-3 of a selection threshold; compacted K/V bit-exact.
"""
import math

import numpy as np
import pytest

from kv_cache_eviction_window_gb300 import datagen
from oracle import kvsel_oracle as O
from tests import gpu_harness as GH

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding

    binding.load()
    yield


def _check_layer(wl, inp, gpu, ora, heads=None):
    for b, (g, o) in enumerate(zip(gpu, ora)):
        n = o["n"]
        assert g["status"] == 0
        fm = O.forced_mask(n, wl.n_sink, wl.n_recent)
        H = wl.h_kv
        hs = range(H) if heads is None else heads
        for h in hs:
            GH.assert_scores_close(g["s_attn"][h], o["s_pool"][h], f"s_attn b{b} h{h}")
            if wl.value_aware:
                GH.assert_scores_close(g["s_val"][h], o["s_val"][h], f"s_val b{b} h{h}")
        if wl.budget_mode == "head":
            B = O.head_budget(n, wl.budget_ratio)
            for h in hs:
                if wl.value_aware:
                    b1 = max(int(math.floor(wl.alpha * B)), int(fm.sum()))
                    t1 = GH.kth_key(o["s_pool"][h], fm, b1)
                    keep1 = np.zeros(n, bool)
                    keep1[O.top_b(o["s_pool"][h], b1, fm)] = True
                    t2 = GH.kth_key(o["s_val"][h], keep1, B)
                    th = [(o["s_pool"][h], t1), (o["s_val"][h], t2)]
                    # the GPU's own scores: stage 1 then stage 2, exactly
                    k1 = GH.topk_mask(g["s_attn"][h], fm, b1)
                    GH.check_topk_property(g["s_val"][h], g["idx"][h], k1, B, f"two-stage b{b} h{h}")
                else:
                    th = [(o["s_pool"][h], GH.kth_key(o["s_pool"][h], fm, B))]
                    GH.check_topk_property(g["s_attn"][h], g["idx"][h], fm, B, f"top-B b{b} h{h}")
                GH.check_selection_near_ties(g["idx"][h], o["idx"][h], fm, n, B, th, f"sel b{b} h{h}")
        else:
            BL = int(math.floor(wl.budget_ratio * n * H))
            fl = int(math.floor(wl.floor_ratio * n))
            assert sum(len(i) for i in g["idx"]) == BL
            fh = min(n, max(fl, int(fm.sum())))
            flat = o["s_pool"].reshape(-1)
            keep = np.zeros((H, n), bool)
            ths = []
            for h in range(H):
                ths.append((o["s_pool"][h], GH.kth_key(o["s_pool"][h], fm, fh)))
                keep[h, O.top_b(o["s_pool"][h], fh, fm)] = True
            tl = GH.kth_key(flat, keep.reshape(-1), BL)
            if wl.value_aware:
                # the layer budget's split over heads (CriticalKV Algorithm 2, line 1): the
                # oracle's allocation, up to entries near the layer threshold
                alloc = O.select_per_layer(o["s_pool"], BL, np.stack([fm] * H), fl)
                for h in range(H):
                    slack = sum(GH.near(x, tl) for x in o["s_pool"][h]) + \
                        sum(GH.near(x, ths[h][1]) for x in o["s_pool"][h])
                    assert abs(len(g["idx"][h]) - len(alloc[h])) <= slack, (b, h, len(g["idx"][h]), len(alloc[h]))
                # then Algorithm 1 within each head's budget (line 8), as in per-head mode
                for h in range(H):
                    Bh = len(g["idx"][h])
                    assert Bh >= fh
                    b1 = max(int(math.floor(wl.alpha * Bh)), int(fm.sum()))
                    t1 = GH.kth_key(o["s_pool"][h], fm, b1)
                    keep1 = np.zeros(n, bool)
                    keep1[O.top_b(o["s_pool"][h], b1, fm)] = True
                    t2 = GH.kth_key(o["s_val"][h], keep1, Bh)
                    want = O.select_two_stage(o["s_pool"][h], o["s_val"][h], Bh, fm, wl.alpha)
                    GH.check_selection_near_ties(g["idx"][h], want, fm, n, Bh,
                                                 [(o["s_pool"][h], t1), (o["s_val"][h], t2)], f"layer va b{b} h{h}")
                    k1 = GH.topk_mask(g["s_attn"][h], fm, b1)
                    GH.check_topk_property(g["s_val"][h], g["idx"][h], k1, Bh, f"layer two-stage b{b} h{h}")
            else:
                for h in range(H):
                    assert len(g["idx"][h]) >= fh
                    GH.check_selection_near_ties(g["idx"][h], o["idx"][h], fm, n, len(g["idx"][h]),
                                                 ths + [(o["s_pool"][h], tl)], f"layer sel b{b} h{h}")
        # compaction is bit-exact given the GPU's own indices
        for h in hs:
            np.testing.assert_array_equal(g["k_out"][h], inp["k"][b][h][g["idx"][h]])
            np.testing.assert_array_equal(g["v_out"][h], inp["v"][b][h][g["idx"][h]])


def test_c1_llama_layer_4k_full():
    wl = datagen.WORKLOADS[1]
    inp = datagen.make_layer(wl, 0)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("n", [1000, 2085])
def test_c2_value_aware_ragged(n):
    wl = datagen.WORKLOADS[2].replace(layers=1)
    inp = datagen.make_layer(wl, 3, n_ctx=n)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("group,window,value_aware", [
    (2, 32, True),    # R = 64: the single-launch scoring with 32-row accumulator halves
    (6, 32, False),   # R = 192: the two-group pass 2 over N = 192
    (4, 64, True),    # R = 256: the largest window the single-launch scoring takes
    (8, 32, False),
])
def test_window_rows_of_the_single_launch_scoring(group, window, value_aware):
    """Window-row counts other than the workloads' 128 that the single cooperative scoring
    launch handles (R a multiple of 64 up to 256), with several tiles per chunk and a
    ragged last tile (CriticalKV §3.4, Algorithm 2: the observation window's softmax)."""
    wl = datagen.WORKLOADS[2].replace(layers=1, group=group, window=window, value_aware=value_aware)
    inp = datagen.make_layer(wl, 11, n_ctx=2085)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("budget,value_aware", [(40, True), (76, False), (200, True)])
def test_sm_budget_sizes_the_kernels_not_the_result(budget, value_aware):
    """kvsel_params.sm_budget only changes how many CTAs the one-per-SM kernels use (key
    chunks of the scoring launch, value-norm CTAs): the layer still matches the oracle.
    A budget above the device's SM count means every SM."""
    wl = datagen.WORKLOADS[2].replace(layers=1, value_aware=value_aware)
    inp = datagen.make_layer(wl, 5, n_ctx=5000)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp, sm_budget=budget)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("n", [1000, 2085])
def test_c2_value_aware_l2_norm(n):
    """nu = ||W_h v||_2 through the d x d Gram matrix (the other distance of CriticalKV
    App. C.3), two-stage selection on it."""
    wl = datagen.WORKLOADS[2].replace(layers=1, value_norm="l2")
    inp = datagen.make_layer(wl, 3, n_ctx=n)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


def test_c4_paged_l2_norm():
    wl = datagen.WORKLOADS[4].replace(batch=3, n_min=300, n_ctx=1500, value_norm="l2", d_model=1024)
    inp = datagen.make_layer(wl, 0)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


def test_c2_per_head_wo_reading():
    wl = datagen.WORKLOADS[2].replace(layers=1, d_model=1024)
    inp = datagen.make_layer(wl, 1, n_ctx=777)
    inp["w_o"] = inp["w_o"]  # [1024][4096]
    ora = O.run_workload_layer(wl, inp, wo_mode="per_head")
    gpu = GH.run_gpu_layer(wl, inp, wo_mode="per_head")
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("n", [1500, 3333])
def test_c3_per_layer_budget(n):
    wl = datagen.WORKLOADS[3].replace(layers=1)
    inp = datagen.make_layer(wl, 0, n_ctx=n)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("n,split", [(1500, False), (3333, False), (3333, True)])
def test_c3_value_aware_per_layer_budget(n, split):
    """Value-aware selection under one budget per layer (CriticalKV Algorithm 2: the layer
    budget split over heads by the pooled attention score, then Algorithm 1 per head) on
    the Qwen2.5-7B layer shape (4 KV heads, group 7, 448 window rows, W_O 3584 x 3584),
    through kvsel_run_layer and through the three split calls."""
    wl = datagen.WORKLOADS[3].replace(value_aware=True, d_model=3584)
    inp = datagen.make_layer(wl, 0, n_ctx=n)
    ora = O.run_workload_layer(wl, inp, compact_out=False)
    gpu = GH.run_gpu_layer(wl, inp, split=split)
    _check_layer(wl, inp, gpu, ora)


def test_c4_paged_ragged_batch():
    wl = datagen.WORKLOADS[4].replace(batch=4, n_min=300, n_ctx=1400)
    inp = datagen.make_layer(wl, 0)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)
    # the same requests from a contiguous (padded) cache give identical results
    gpu2 = GH.run_gpu_layer(wl, inp, paged=False)
    for a, b in zip(gpu, gpu2):
        np.testing.assert_array_equal(a["s_attn"], b["s_attn"])
        for h in range(wl.h_kv):
            np.testing.assert_array_equal(a["idx"][h], b["idx"][h])


@pytest.mark.parametrize("reduce,pool,causal", [("sum", "none", False), ("max", "max", True),
                                                 ("mean", "avg", True)])
def test_reductions_and_pooling(reduce, pool, causal):
    wl = datagen.WORKLOADS[1].replace(reduce=reduce, pool=pool, pool_kernel=5, causal=causal,
                                      h_kv=2, n_ctx=1111)
    inp = datagen.make_layer(wl, 0, n_ctx=1111)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("cid,n,kw", [
    (1, 1111, dict(pool="max", pool_kernel=7)),
    (2, 1500, dict()),                                   # value-aware, two-stage, avg pooling
    (3, 1333, dict()),                                   # per-layer budget with floors
    (1, 1111, dict(pool="avg", pool_kernel=67)),         # halo wider than the fused staging
])
def test_split_calls_match_run_layer(cid, n, kw):
    """kvsel_score + kvsel_select + kvsel_compact give exactly what kvsel_run_layer gives
    (the latter pools inside the selection), and both match the oracle."""
    wl = datagen.WORKLOADS[cid].replace(**kw)
    if cid == 2:
        wl = wl.replace(layers=1, h_kv=2, d_model=1024)
    inp = datagen.make_layer(wl, 0, n_ctx=n)
    ora = O.run_workload_layer(wl, inp)
    fused = GH.run_gpu_layer(wl, inp)
    split = GH.run_gpu_layer(wl, inp, split=True)
    _check_layer(wl, inp, fused, ora)
    for a, b in zip(fused, split):
        np.testing.assert_array_equal(a["s_attn"], b["s_attn"])
        if a["s_val"] is not None:
            np.testing.assert_array_equal(a["s_val"], b["s_val"])
        for h in range(wl.h_kv):
            np.testing.assert_array_equal(a["idx"][h], b["idx"][h])
            np.testing.assert_array_equal(a["k_out"][h], b["k_out"][h])
            np.testing.assert_array_equal(a["v_out"][h], b["v_out"][h])


def test_two_stage_with_empty_first_stage():
    """floor(alpha * B) = 0 and no forced entries: stage 1 takes nothing, so the single
    kept entry per head is the value-aware argmax (radix selection of zero entries)."""
    wl = datagen.WORKLOADS[2].replace(layers=1, h_kv=2, d_model=512, n_sink=0, n_recent=0, budget_ratio=0.001)
    inp = datagen.make_layer(wl, 0, n_ctx=1000)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    for h in range(2):
        GH.assert_scores_close(gpu[0]["s_val"][h], ora[0]["s_val"][h], f"s_val h{h}")
        assert len(gpu[0]["idx"][h]) == 1 and len(ora[0]["idx"][h]) == 1
        sv = ora[0]["s_val"][h]
        assert sv[gpu[0]["idx"][h][0]] >= sv.max() * (1 - GH.SEL_RTOL)


def test_budget_equals_n_identity():
    wl = datagen.WORKLOADS[1].replace(budget_ratio=1.0, h_kv=2)
    inp = datagen.make_layer(wl, 0, n_ctx=600)
    gpu = GH.run_gpu_layer(wl, inp)
    for h in range(2):
        np.testing.assert_array_equal(gpu[0]["idx"][h], np.arange(600))
        np.testing.assert_array_equal(gpu[0]["k_out"][h], inp["k"][0][h])


def test_minimal_context_equals_window():
    wl = datagen.WORKLOADS[1].replace(h_kv=1, n_recent=32, n_sink=4, budget_ratio=1.0)
    inp = datagen.make_layer(wl, 0, n_ctx=32)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("n", [1000, 2048])
def test_c5_query_agnostic(n):
    """KVzip maximum cross-attention score: all G*n positions as queries, non-causal,
    max over queries and group heads, one budget per layer."""
    wl = datagen.WORKLOADS[5].replace(h_kv=4)
    inp = datagen.make_layer(wl, 0, n_ctx=n)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("n", [1000, 2048])
def test_c5_logit_scores_and_head_scores(n):
    """KVzip-logit (softmax-free): the maximum scaled dot product over all G*n query rows,
    one budget per layer; and head-level scores (max over the sequence) of those scores."""
    import torch
    from kv_cache_eviction_window_gb300 import binding as B

    wl = datagen.WORKLOADS[5].replace(h_kv=4, reduce="max_logit")
    inp = datagen.make_layer(wl, 0, n_ctx=n)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)
    p = B.params_from_workload(wl, n_ctx=n)
    s = torch.from_numpy(np.concatenate([gpu[0]["s_attn"][h] for h in range(wl.h_kv)])).cuda()
    hs = torch.empty(wl.h_kv, dtype=torch.float32, device="cuda")
    B.kvsel_head_scores(p, s, hs)
    hs = hs.cpu().numpy()
    np.testing.assert_array_equal(hs, [gpu[0]["s_attn"][h].max() for h in range(wl.h_kv)])
    GH.assert_scores_close(hs, O.head_scores(ora[0]["s_pool"]), "head scores")


def test_head_scores_ragged_batch():
    """Head scores over a packed ragged batch (per request and head)."""
    import torch
    from kv_cache_eviction_window_gb300 import binding as B

    wl = datagen.WORKLOADS[4].replace(batch=5, n_min=100, n_ctx=700)
    lens = datagen.context_lengths(wl)
    p = B.params_from_workload(wl, n_ctx_per_req=lens)
    rng = np.random.default_rng(3)
    parts = [rng.standard_normal((wl.h_kv, n)).astype(np.float32) for n in lens]
    s = torch.from_numpy(np.concatenate([x.reshape(-1) for x in parts])).cuda()
    hs = torch.empty(len(lens) * wl.h_kv, dtype=torch.float32, device="cuda")
    B.kvsel_head_scores(p, s, hs)
    want = np.concatenate([x.max(axis=1) for x in parts])
    np.testing.assert_array_equal(hs.cpu().numpy(), want)


# ---------------------------------------------------------------------- full size
def test_c2_full_layer_plain_full_oracle():
    """Llama-3.1-8B layer, n = 32768, attention score only: every pooled score and every
    head's kept set against the full oracle."""
    wl = datagen.WORKLOADS[2].replace(value_aware=False)
    inp = datagen.make_layer(wl, 0)
    ora = O.run_workload_layer(wl, inp, compact_out=False)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)
    # the benchmark's plain-path configuration: overlapping calls sized for a twelfth of
    # the SMs (two scoring launches of two long chunks per head, 2-CTA selection
    # clusters), and for a fifth and half of them (4-CTA clusters at half)
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for budget in (sms // 12, sms // 5, sms // 2):
        gpu = GH.run_gpu_layer(wl, inp, concurrent=True, sm_budget=budget)
        _check_layer(wl, inp, gpu, ora)


def test_c2_full_layer_value_aware_full_oracle():
    """The benchmark's layer (Llama-3.1-8B, n = 32768, value-aware two-stage selection)
    against the full oracle: s_attn and s_val on every token of every head (the oracle's
    ||W_h v||_1 for all 8 x 32768 tokens), each head's kept set against the oracle's own
    two-stage selection (differences only at near-ties of either stage's threshold) and as
    the exact two-stage top-B of the GPU's scores, and the compacted rows bit for bit."""
    wl = datagen.WORKLOADS[2]
    inp = datagen.make_layer(wl, 0)
    ora = O.run_workload_layer(wl, inp, compact_out=False)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)
    # the benchmark's headline configuration: overlapping calls on every SM (two scoring
    # launches, 4-CTA selection clusters)
    gpu = GH.run_gpu_layer(wl, inp, concurrent=True)
    _check_layer(wl, inp, gpu, ora)


def test_c3_full_layer():
    """Qwen2.5-7B layer, n = 131072, 448 window rows per head, per-layer budget."""
    wl = datagen.WORKLOADS[3]
    inp = datagen.make_layer(wl, 0)
    ora = O.run_workload_layer(wl, inp, compact_out=False)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


# ---------------------------------------------------------------------- device status
def test_bounded_wait_timeout_reports_status():
    """A wait budget of 1 cycle (kvsel_params.wait_cycles) makes the pipeline waits give
    up: the kernels end with KVSEL_ETIMEOUT in the status word and the context stays
    usable.  The budget is a per-call parameter, so the next call with the default runs
    normally."""
    from kv_cache_eviction_window_gb300 import binding as B

    wl = datagen.WORKLOADS[1].replace(h_kv=2)
    inp = datagen.make_layer(wl, 0, n_ctx=2048)
    out = GH.run_gpu_layer(wl, inp, wait_cycles=1)
    assert out[0]["status"] == B.KVSEL_ETIMEOUT
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


def test_c5_logit_full_layer_sampled_keys():
    """KVzip-logit at n = 32768: 12 keys per head checked exactly against the maximum over
    all 262144 query rows, every key against a sampled-row lower bound, and the kept set
    is exactly the layer top-B of the GPU's own scores."""
    wl = datagen.WORKLOADS[5].replace(reduce="max_logit")
    inp = datagen.make_layer(wl, 0)
    gpu = GH.run_gpu_layer(wl, inp)[0]
    n, H = wl.n_ctx, wl.h_kv
    rng = np.random.default_rng(6)
    k = O.bf16_to_f64(inp["k"][0])
    for h in range(H):
        s = gpu["s_attn"][h].astype(np.float64)
        q = O.bf16_to_f64(inp["q"][0][h])                        # [G][n][d]
        keys = rng.choice(n, size=12, replace=False)
        exact = O.query_agnostic_logit_scores(q, k[h][keys])
        GH.assert_scores_close(s[keys], exact, f"head {h} sampled keys")
        pos = rng.choice(n, size=6, replace=False)
        lower = O.query_agnostic_logit_scores(q[:, pos, :], k[h])
        assert np.all(s >= lower - 1e-4 * np.abs(lower).max()), f"head {h}"
    fm = O.forced_mask(n, wl.n_sink, wl.n_recent)
    BL = int(math.floor(wl.budget_ratio * n * H))
    flat = np.concatenate([gpu["s_attn"][h] for h in range(H)])
    kept = np.concatenate([np.asarray(gpu["idx"][h]) + h * n for h in range(H)])
    GH.check_topk_property(flat, np.sort(kept), np.tile(fm, H), BL, "C5-logit layer top-B")


def test_c5_full_layer_sampled_rows():
    """Llama-3.1-70B layer shape, n = 32768 (262144 query rows per KV head).  The oracle
    cannot form every row's normaliser at this size, so: every score is a probability,
    it is at least the oracle's score over a sample of 48 query rows per head (a max over
    a subset), and the kept set is exactly the layer top-B of the GPU's own scores."""
    wl = datagen.WORKLOADS[5]
    inp = datagen.make_layer(wl, 0)
    gpu = GH.run_gpu_layer(wl, inp)[0]
    n, H = wl.n_ctx, wl.h_kv
    rng = np.random.default_rng(5)
    k = O.bf16_to_f64(inp["k"][0])
    for h in range(H):
        s = gpu["s_attn"][h].astype(np.float64)
        assert np.all(s > 0) and np.all(s <= 1.0 + 1e-6)
        pos = rng.choice(n, size=6, replace=False)
        qs = O.bf16_to_f64(inp["q"][0][h][:, pos, :])          # [G][6][d]
        lower = O.query_agnostic_scores(qs, k[h])
        assert np.all(s >= lower * (1 - GH.RTOL) - GH.ATOL_FRAC * lower.max()), f"head {h}"
    fm = O.forced_mask(n, wl.n_sink, wl.n_recent)
    BL = int(math.floor(wl.budget_ratio * n * H))
    flat = np.concatenate([gpu["s_attn"][h] for h in range(H)])
    kept = np.concatenate([np.asarray(gpu["idx"][h]) + h * n for h in range(H)])
    GH.check_topk_property(flat, np.sort(kept), np.tile(fm, H), BL, "C5 layer top-B")


def test_select_after_a_smaller_cluster_query():
    """A long selection, then a short one (a new cluster-size query at a smaller shared-
    memory size), then the long one again: the second long launch must still get its
    shared-memory limit (the query may not lower a limit the launch path relies on)."""
    import torch
    from kv_cache_eviction_window_gb300 import binding as B

    def run(n, seed):
        s = datagen.random_scores(1, n, seed)[0]
        p = B.make_params(h_kv=1, group=4, n_ctx=n, window=32, budget_ratio=0.4, n_sink=4, n_recent=32)
        buf = B.LayerBuffers(p)
        buf.s_attn.copy_(torch.from_numpy(s))
        B.kvsel_select(p, buf.s_attn, None, buf.idx, buf.counts, buf.offsets, buf.ws)
        torch.cuda.synchronize()
        fm = O.forced_mask(n, 4, 32)
        want = O.top_b(s.astype(np.float64), O.head_budget(n, 0.4), fm)
        np.testing.assert_array_equal(buf.idx[:len(want)].cpu().numpy(), want)

    run(131072, 1)
    run(1000 + 17, 2)
    run(131072, 3)


def test_two_stage_select_more_entries_per_cta_than_registers_hold():
    """One KV head of 70000 keys: its selection cluster of 16 CTAs gives each CTA 4375
    entries, more than its threads keep in registers (8 x 512), so the value-aware keys of
    the second stage are read back from the scores the selection kernel wrote."""
    wl = datagen.WORKLOADS[2].replace(layers=1, h_kv=1, d_model=512)
    inp = datagen.make_layer(wl, 0, n_ctx=70000)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)


def test_compact_out_of_range_index_is_zeroed_and_flagged():
    """kvsel_compact with two out-of-range indices among valid ones: the valid rows are
    bit-exact copies, the bad rows come out as zeros, and the status word reports it."""
    import torch
    from kv_cache_eviction_window_gb300 import binding as B

    wl = datagen.WORKLOADS[2].replace(layers=1, h_kv=2)
    n = 700
    inp = datagen.make_layer(wl, 0, n_ctx=n)
    p = B.params_from_workload(wl, n_ctx=n)
    kc, vc = np.stack(inp["k"]), np.stack(inp["v"])   # [1][H][n][d]
    kt, vt = GH.torch_bf16(kc), GH.torch_bf16(vc)
    kv = B.make_kv_contiguous(kt, vt)
    rng = np.random.default_rng(3)
    per_head = [np.sort(rng.choice(n, size=150, replace=False)).astype(np.int32) for _ in range(wl.h_kv)]
    per_head[0][10] = n + 5      # past the context
    per_head[1][77] = -3         # negative
    flat = np.concatenate(per_head)
    counts = np.array([len(x) for x in per_head], np.int32)
    offsets = np.array([0, len(per_head[0])], np.int64)
    ws = torch.zeros(B.kvsel_workspace_size(p) // 4 + 64, dtype=torch.int32, device="cuda")
    B.kvsel_workspace_init(ws)
    k_out = torch.full((len(flat), wl.head_dim), 7.0, dtype=torch.bfloat16, device="cuda")
    v_out = torch.full((len(flat), wl.head_dim), 7.0, dtype=torch.bfloat16, device="cuda")
    B.kvsel_compact(p, kv, torch.from_numpy(flat).cuda(), torch.from_numpy(counts).cuda(),
                    torch.from_numpy(offsets).cuda(), k_out, v_out, ws)
    torch.cuda.synchronize()
    assert B.kvsel_get_device_status(ws) == B.KVSEL_EDEVICE
    ko = k_out.cpu().view(torch.int16).numpy().view(np.uint16)
    vo = v_out.cpu().view(torch.int16).numpy().view(np.uint16)
    for h in range(wl.h_kv):
        o = int(offsets[h])
        for r, i in enumerate(per_head[h]):
            if 0 <= i < n:
                np.testing.assert_array_equal(ko[o + r], kc[0, h, i])
                np.testing.assert_array_equal(vo[o + r], vc[0, h, i])
            else:
                assert not ko[o + r].any() and not vo[o + r].any(), f"head {h} row {r}"


def test_ex2_probe_rate_is_plausible():
    """The benchmark's exponential-unit probe: a positive rate per SM clock within what an
    SM can issue, and a device rate consistent with it at a clock between 0.5 and 3 GHz."""
    import torch

    import bench

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_clk, per_s = bench.ex2_probe_rate(torch.empty(16 * sms, dtype=torch.uint8, device="cuda"))
    assert 4.0 <= per_clk <= 128.0, per_clk
    ghz = per_s / (per_clk * sms) / 1e9
    assert 0.5 <= ghz <= 3.0, ghz
    with pytest.raises(RuntimeError, match="returned -4"):
        bench.ex2_probe_rate(torch.empty(16 * sms - 16, dtype=torch.uint8, device="cuda"))


def test_c4_full_batch_full_oracle():
    """The ragged serving batch at full size: 16 requests of 2048-65536 tokens in a paged
    cache (block 16, shuffled block table), value-aware.  Every request and head against
    the full oracle: pooled and value-aware scores on every token, the kept sets (near-ties
    only) and the compacted rows bit for bit."""
    wl = datagen.WORKLOADS[4]
    inp = datagen.make_layer(wl, 0)
    gpu = GH.run_gpu_layer(wl, inp)
    ora = O.run_workload_layer(wl, inp, compact_out=False)
    _check_layer(wl, inp, gpu, ora)


def test_c2_full_layer_l2_norm_full_oracle():
    """The L2 value norm (the d x d Gram path) on the 32K Llama-3.1-8B layer against the
    full oracle (||W_h v||_2 for every token of every head): scores, kept sets and the
    compacted rows."""
    wl = datagen.WORKLOADS[2].replace(value_norm="l2")
    inp = datagen.make_layer(wl, 0)
    gpu = GH.run_gpu_layer(wl, inp)
    ora = O.run_workload_layer(wl, inp, compact_out=False)
    _check_layer(wl, inp, gpu, ora)


def test_c5_softmax_exact_at_the_full_size_split():
    """KVzip's softmax score, exact against the full oracle, on a layer whose work split
    matches the 70B-shaped n = 32768 layer: the same number of query-row slices per key
    block (4, merged by atomic max), whole 256-key blocks and whole 512-row LSE blocks
    (32 KV heads x 3328 keys, group 8, 26624 query rows per head)."""
    from kv_cache_eviction_window_gb300 import binding as B

    full = datagen.WORKLOADS[5]
    kb_full, rs_full = B.kvsel_query_agnostic_split(B.params_from_workload(full))
    wl = full.replace(h_kv=32)
    n = 3328
    kb, rs = B.kvsel_query_agnostic_split(B.params_from_workload(wl, n_ctx=n))
    assert rs == rs_full and rs > 1, (rs, rs_full)
    assert kb * 256 == n and kb_full * 256 == full.n_ctx
    assert (wl.group * n) % 512 == 0 and (full.group * full.n_ctx) % 512 == 0
    inp = datagen.make_layer(wl, 0, n_ctx=n)
    ora = O.run_workload_layer(wl, inp, compact_out=False)
    gpu = GH.run_gpu_layer(wl, inp)
    _check_layer(wl, inp, gpu, ora)
