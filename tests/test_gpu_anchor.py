"""AnchorKV anchors on the GPU against the fp64 oracle ("AnchorKV: Anchor-Residual KV
Cache Compression", §3.1-§3.2, §4.1).

Anchor selection is compared as a kept set (GPU and oracle may differ only through
stage-1 near-ties of the pooled score); the anchor rows are bit-exact copies; the
projection is compared slot by slot: the GPU's slot must reach the oracle's largest
cosine within COS_TOL (exact agreement is also counted), and gamma must match the
oracle's coefficient for that slot.
"""
import numpy as np
import pytest

from kv_cache_eviction_window_gb300 import datagen
from tests import gpu_harness as GH

pytestmark = pytest.mark.gpu

# fp32 dot products of bf16 inputs: |error| ~ 1e-6 |x| |a|, so cosines carry ~1e-6
COS_TOL = 2e-5
GAMMA_RTOL = 1e-5


def _kv_for(wl, inp, paged):
    import torch
    from kv_cache_eviction_window_gb300 import binding as B

    lens = inp["n_ctx"]
    if paged:
        pg = inp["paged"]
        kp, vp = GH.torch_bf16(pg["k_pool"]), GH.torch_bf16(pg["v_pool"])
        table = torch.from_numpy(pg["block_table"]).cuda()
        return B.make_kv_paged(kp, vp, table), (kp, vp, table)
    H, d = wl.h_kv, wl.head_dim
    nmax = max(lens)
    kc = np.zeros((len(lens), H, nmax, d), np.uint16)
    vc = np.zeros((len(lens), H, nmax, d), np.uint16)
    for b in range(len(lens)):
        kc[b, :, :lens[b]] = inp["k"][b]
        vc[b, :, :lens[b]] = inp["v"][b]
    kt, vt = GH.torch_bf16(kc), GH.torch_bf16(vc)
    return B.make_kv_contiguous(kt, vt), (kt, vt)


def _unpack(wl, buf, lens):
    import torch

    H = wl.h_kv
    s_attn = buf.s_attn.cpu().numpy()
    idx, counts, offsets = buf.idx.cpu().numpy(), buf.counts.cpu().numpy(), buf.offsets.cpu().numpy()
    k_out = buf.k_out.cpu().view(torch.int16).numpy().view(np.uint16)
    v_out = buf.v_out.cpu().view(torch.int16).numpy().view(np.uint16)
    sk, gk = buf.slot_k.cpu().numpy(), buf.gamma_k.cpu().numpy()
    sv, gv = buf.slot_v.cpu().numpy(), buf.gamma_v.cpu().numpy()
    out, so = [], 0
    for b, n in enumerate(lens):
        r = dict(n=n, s_attn=s_attn[so:so + H * n].reshape(H, n))
        for name, arr in (("slot_k", sk), ("gamma_k", gk), ("slot_v", sv), ("gamma_v", gv)):
            r[name] = arr[so:so + H * n].reshape(H, n)
        so += H * n
        r["anchors"], r["k_out"], r["v_out"] = [], [], []
        for h in range(H):
            c, o = int(counts[b * H + h]), int(offsets[b * H + h])
            r["anchors"].append(idx[o:o + c].astype(np.int64))
            r["k_out"].append(k_out[o:o + c])
            r["v_out"].append(v_out[o:o + c])
        out.append(r)
    return out


def run_gpu_anchors(wl, inp, paged=False):
    """kvsel_run_anchors on one layer of seeded inputs."""
    import torch
    from kv_cache_eviction_window_gb300 import binding as B

    lens = inp["n_ctx"]
    p = B.params_from_workload(wl, n_ctx_per_req=lens if len(lens) > 1 else None, n_ctx=lens[0])
    q = GH.torch_bf16(inp["q"])
    kv, keep = _kv_for(wl, inp, paged)
    rand = torch.from_numpy(np.concatenate([r.reshape(-1) for r in inp["rand"]]).astype(np.float32)).cuda()
    buf = B.LayerBuffers(p)
    B.kvsel_run_anchors(p, q, kv, rand, buf.s_attn, buf.idx, buf.counts, buf.offsets, buf.k_out, buf.v_out,
                        buf.slot_k, buf.gamma_k, buf.slot_v, buf.gamma_v, buf.ws)
    torch.cuda.synchronize()
    status = B.kvsel_get_device_status(buf.ws)
    del keep
    assert status == 0, f"device status {status}"
    return _unpack(wl, buf, lens)


def run_gpu_projection(wl, inp, anchors, paged=False):
    """kvsel_compact + kvsel_anchor_project with a given anchor list per (request, head)."""
    import torch
    from kv_cache_eviction_window_gb300 import binding as B

    lens = inp["n_ctx"]
    p = B.params_from_workload(wl, n_ctx_per_req=lens if len(lens) > 1 else None, n_ctx=lens[0])
    kv, keep = _kv_for(wl, inp, paged)
    buf = B.LayerBuffers(p)
    flat = np.concatenate([a for req in anchors for a in req]).astype(np.int32)
    cnt = np.array([len(a) for req in anchors for a in req], np.int32)
    off = np.concatenate([[0], np.cumsum(cnt)[:-1]]).astype(np.int64)
    assert len(flat) <= buf.idx.numel()
    buf.idx[:len(flat)].copy_(torch.from_numpy(flat))
    buf.counts.copy_(torch.from_numpy(cnt))
    buf.offsets.copy_(torch.from_numpy(off))
    B.kvsel_compact(p, kv, buf.idx, buf.counts, buf.offsets, buf.k_out, buf.v_out, buf.ws)
    B.kvsel_anchor_project(p, kv, buf.k_out, buf.v_out, buf.idx, buf.counts, buf.offsets, buf.slot_k, buf.gamma_k,
                           buf.slot_v, buf.gamma_v, buf.ws)
    torch.cuda.synchronize()
    status = B.kvsel_get_device_status(buf.ws)
    del keep
    assert status == 0, f"device status {status}"
    return _unpack(wl, buf, lens)


def check_projection(x_bits, anchors, slot, gamma, rows, what):
    """Compare the GPU's (slot, gamma) of positions `rows` of one (request, head, side)
    with the oracle's nearest-anchor projection; returns the exact-slot agreement."""
    from oracle import anchor_oracle as AO
    from oracle import kvsel_oracle as O

    x = O.bf16_to_f64(x_bits)
    anchors = np.asarray(anchors, np.int64)
    k = len(anchors)
    rows = np.asarray(rows, np.int64)
    # the oracle on [anchor rows; sampled rows]: slots 0..k-1 are the anchors themselves
    sub = np.concatenate([x[anchors], x[rows]])
    o_slot, o_gamma, cos = AO.anchor_project(sub, np.arange(k))
    o_slot, o_gamma, cos = o_slot[k:], o_gamma[k:], cos[k:]
    is_anchor = np.isin(rows, anchors)
    g_slot = slot[rows].astype(np.int64)
    g_gamma = gamma[rows].astype(np.float64)
    if k == 0:
        assert (g_slot == 0).all() and (g_gamma == 0).all(), what
        return 1.0
    assert ((g_slot >= 0) & (g_slot < k)).all(), f"{what}: slot out of range"
    # anchors: themselves, exactly
    own = np.searchsorted(anchors, rows[is_anchor])
    assert (g_slot[is_anchor] == own).all() and (g_gamma[is_anchor] == 1.0).all(), f"{what}: anchor not itself"
    na = ~is_anchor
    r = np.arange(len(rows))[na]
    best = cos[r].max(axis=1)
    got = cos[r, g_slot[na]]
    bad = got < best - COS_TOL
    assert not bad.any(), f"{what}: {bad.sum()} slots below the best cosine (worst gap {np.max(best - got)})"
    a = x[anchors][g_slot[na]]
    xr = x[rows][na]
    a2 = (a * a).sum(1)
    ref = np.divide((xr * a).sum(1), a2, out=np.zeros(len(r)), where=a2 > 0)
    scale = np.sqrt((xr * xr).sum(1)) / np.sqrt(np.where(a2 > 0, a2, 1.0))
    err = np.abs(g_gamma[na] - ref)
    tol = GAMMA_RTOL * (np.abs(ref) + scale)
    assert (err <= tol).all(), f"{what}: gamma off by {np.max(err / tol)} x tolerance"
    return float(np.mean(g_slot[na] == o_slot[na])) if na.any() else 1.0


def _compare_anchor_run(wl, inp, gpu, ora, sample=None, min_agree=0.999):
    rng = np.random.default_rng(0)
    for b, (g, o) in enumerate(zip(gpu, ora)):
        n = g["n"]
        GH.assert_scores_close(g["s_attn"], o["s_pool"], f"req {b} pooled score")
        fm = np.zeros(n, bool)
        fm[:min(wl.n_sink, n)] = True
        if wl.n_recent:
            fm[max(n - wl.n_recent, 0):] = True
        for h in range(wl.h_kv):
            ga, oa = g["anchors"][h], o["anchors"][h]
            assert len(ga) == o["k"], f"req {b} head {h}: {len(ga)} anchors, expected {o['k']}"
            assert np.all(np.diff(ga) > 0) and (len(ga) == 0 or (ga[0] >= 0 and ga[-1] < n))
            # rows are bit-exact copies of the anchors' K and V
            assert np.array_equal(g["k_out"][h], inp["k"][b][h][ga]), f"req {b} head {h}: anchor K rows"
            assert np.array_equal(g["v_out"][h], inp["v"][b][h][ga]), f"req {b} head {h}: anchor V rows"
            if not np.array_equal(ga, oa):
                # only through stage-1 near-ties of the pooled score
                nf = int(fm.sum())
                k1 = nf + int(np.floor(wl.alpha * (o["k"] - nf)))
                t1 = GH.kth_key(o["s_pool"][h], fm, k1)
                diff = set(ga.tolist()) ^ set(oa.tolist())
                assert any(GH.near(o["s_pool"][h][i], t1) for i in diff), (
                    f"req {b} head {h}: anchor sets differ without a stage-1 near-tie")
                continue
            rows = np.arange(n) if sample is None or n <= sample else np.sort(rng.choice(n, sample, replace=False))
            rows = np.union1d(rows, ga[: min(len(ga), 64)])
            for side in ("k", "v"):
                agree = check_projection(inp[side][b][h], ga, g["slot_" + side][h], g["gamma_" + side][h], rows,
                                         f"req {b} head {h} {side}")
                assert agree >= min_agree, f"req {b} head {h} {side}: exact slot agreement {agree}"


def test_anchor_small_end_to_end():
    # n = 9000: k = 70 = 32 recent + 26 by score + 12 random
    from oracle import anchor_oracle as AO

    wl = datagen.WORKLOADS[6].replace(h_kv=2)
    inp = datagen.make_layer(wl, 0, n_ctx=9000)
    gpu = run_gpu_anchors(wl, inp)
    ora = AO.run_anchor_workload_layer(wl, inp, project=False)
    _compare_anchor_run(wl, inp, gpu, ora)


def test_anchor_ragged_paged_batch():
    # ragged paged batch; budget 1/64 and a recent window of 8 leave free slots at these n
    from oracle import anchor_oracle as AO

    wl = datagen.WORKLOADS[6].replace(batch=3, n_min=300, n_ctx=2500, paged=True, block_size=16, n_recent=8,
                                      budget_ratio=1.0 / 64)
    inp = datagen.make_layer(wl, 0)
    gpu = run_gpu_anchors(wl, inp, paged=True)
    ora = AO.run_anchor_workload_layer(wl, inp, project=False)
    _compare_anchor_run(wl, inp, gpu, ora)


def test_anchor_projection_given_anchors_multichunk():
    # 600 anchors per head: three chunks of up to 256 (the multi-chunk path), ragged tail
    wl = datagen.WORKLOADS[6].replace(h_kv=2, budget_ratio=0.1)
    n = 6000
    inp = datagen.make_layer(wl, 0, n_ctx=n)
    anchors = [[datagen.anchor_positions(n, 600, wl.n_recent, 100 + h) for h in range(2)]]
    gpu = run_gpu_projection(wl, inp, anchors)
    for h in range(2):
        assert np.array_equal(gpu[0]["anchors"][h], anchors[0][h])
        for side in ("k", "v"):
            agree = check_projection(inp[side][0][h], anchors[0][h], gpu[0]["slot_" + side][h],
                                     gpu[0]["gamma_" + side][h], np.arange(n), f"head {h} {side}")
            assert agree >= 0.999


def test_anchor_projection_full_size_sampled():
    # the benchmark's shape: Llama-3.1-8B, n = 32768, 256 anchors per head (given)
    wl = datagen.WORKLOADS[6]
    n = wl.n_ctx
    inp = datagen.make_layer(wl, 0)
    anchors = [[datagen.anchor_positions(n, n // 128, wl.n_recent, 200 + h) for h in range(wl.h_kv)]]
    gpu = run_gpu_projection(wl, inp, anchors)
    rng = np.random.default_rng(1)
    for h in range(wl.h_kv):
        rows = np.union1d(np.sort(rng.choice(n, 1500, replace=False)), np.arange(n - 200, n))
        for side in ("k", "v"):
            agree = check_projection(inp[side][0][h], anchors[0][h], gpu[0]["slot_" + side][h],
                                     gpu[0]["gamma_" + side][h], rows, f"head {h} {side}")
            assert agree >= 0.999


def test_anchor_full_size_end_to_end_sampled():
    from oracle import anchor_oracle as AO

    wl = datagen.WORKLOADS[6]
    inp = datagen.make_layer(wl, 0)
    gpu = run_gpu_anchors(wl, inp)
    ora = AO.run_anchor_workload_layer(wl, inp, project=False)
    _compare_anchor_run(wl, inp, gpu, ora, sample=1500)


def test_anchor_degenerate_no_anchors_and_all_forced():
    # n = 100 with no recent window: k = floor(100/128) = 0 -> slot 0, gamma 0 everywhere;
    # n = 4096: k = 32 = the recent window (no free slot)
    from oracle import anchor_oracle as AO

    wl = datagen.WORKLOADS[6].replace(h_kv=2, window=8, n_recent=0)
    inp = datagen.make_layer(wl, 0, n_ctx=100)
    gpu = run_gpu_anchors(wl, inp)
    for h in range(2):
        assert len(gpu[0]["anchors"][h]) == 0
        assert (gpu[0]["slot_k"][h] == 0).all() and (gpu[0]["gamma_v"][h] == 0).all()
    wl2 = datagen.WORKLOADS[6].replace(h_kv=2)
    inp2 = datagen.make_layer(wl2, 0, n_ctx=4096)
    gpu2 = run_gpu_anchors(wl2, inp2)
    ora2 = AO.run_anchor_workload_layer(wl2, inp2, project=False)
    _compare_anchor_run(wl2, inp2, gpu2, ora2)


def test_anchor_selection_more_entries_per_cta_than_registers_hold():
    """One KV head of 70000 keys: each CTA of the 16-CTA selection cluster holds 4375
    entries, so the random keys of the second stage are read back from memory rather than
    kept in registers."""
    from oracle import anchor_oracle as AO

    wl = datagen.WORKLOADS[6].replace(h_kv=1)
    inp = datagen.make_layer(wl, 0, n_ctx=70000)
    gpu = run_gpu_anchors(wl, inp)
    ora = AO.run_anchor_workload_layer(wl, inp, project=False)
    _compare_anchor_run(wl, inp, gpu, ora, sample=1500)
