"""Helpers shared by the GPU tests: upload seeded inputs, run the CUDA path through the
C ABI, and compare with the oracle under the stated tolerances.  Importing this module
does not need a GPU."""
import numpy as np

# Score tolerance: |gpu - oracle| <= RTOL*|oracle| + ATOL_FRAC*max|oracle| (per (b, h)).
# RTOL is the 1e-3 relative bound for fp32 accumulation of bf16 inputs; the absolute
# floor covers entries flushed to zero (denormal exponentials) on the GPU.
RTOL = 1e-3
ATOL_FRAC = 1e-7
# Selection: entries may differ only where the oracle's score lies within SEL_RTOL
# (relative) of the selection threshold.
SEL_RTOL = 1e-3


def torch_bf16(u16, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(device)


def run_gpu_layer(wl, inp, paged=None, ws_pad=0, split=False, **override):
    """Run kvsel_run_layer on one layer of seeded inputs; return numpy outputs per request.
    With split=True the three stages are called one by one (kvsel_score, kvsel_select,
    kvsel_compact) instead, which pools in its own kernel rather than inside the selection."""
    import torch
    from kv_cache_eviction_window_gb300 import binding as B

    lens = inp["n_ctx"]
    bsz = len(lens)
    p = B.params_from_workload(wl, n_ctx_per_req=lens if bsz > 1 else None,
                               n_ctx=lens[0], **override)
    q = torch_bf16(inp["q"])
    use_paged = wl.paged if paged is None else paged
    if use_paged:
        pg = inp["paged"]
        kp, vp = torch_bf16(pg["k_pool"]), torch_bf16(pg["v_pool"])
        table = torch.from_numpy(pg["block_table"]).cuda()
        kv = B.make_kv_paged(kp, vp, table)
        keep = (kp, vp, table)
    else:
        H, d = wl.h_kv, wl.head_dim
        nmax = max(lens)
        kc = np.zeros((bsz, H, nmax, d), np.uint16)
        vc = np.zeros((bsz, H, nmax, d), np.uint16)
        for b in range(bsz):
            kc[b, :, :lens[b]] = inp["k"][b]
            vc[b, :, :lens[b]] = inp["v"][b]
        kt, vt = torch_bf16(kc), torch_bf16(vc)
        kv = B.make_kv_contiguous(kt, vt)
        keep = (kt, vt)
    w_o = torch_bf16(inp["w_o"]) if inp["w_o"] is not None and p.value_aware else None
    buf = B.LayerBuffers(p)
    if split:
        B.kvsel_score(p, q, kv, w_o, buf.s_attn, buf.s_val, buf.ws)
        B.kvsel_select(p, buf.s_attn, buf.s_val, buf.idx, buf.counts, buf.offsets, buf.ws)
        B.kvsel_compact(p, kv, buf.idx, buf.counts, buf.offsets, buf.k_out, buf.v_out, buf.ws)
    else:
        B.kvsel_run_layer(p, q, kv, w_o, buf.s_attn, buf.s_val, buf.idx, buf.counts, buf.offsets, buf.k_out,
                          buf.v_out, buf.ws)
    torch.cuda.synchronize()
    status = B.kvsel_get_device_status(buf.ws)
    del keep
    return unpack(wl, p, buf, lens, status)


def unpack(wl, p, buf, lens, status=0):
    H = wl.h_kv
    s_attn = buf.s_attn.cpu().numpy()
    s_val = buf.s_val.cpu().numpy() if buf.s_val is not None else None
    idx = buf.idx.cpu().numpy()
    counts = buf.counts.cpu().numpy()
    offsets = buf.offsets.cpu().numpy()
    import torch

    k_out = buf.k_out.cpu().view(torch.int16).numpy().view(np.uint16)
    v_out = buf.v_out.cpu().view(torch.int16).numpy().view(np.uint16)
    out = []
    so = 0
    for b, n in enumerate(lens):
        r = dict(n=n, status=status)
        r["s_attn"] = s_attn[so:so + H * n].reshape(H, n)
        r["s_val"] = s_val[so:so + H * n].reshape(H, n) if s_val is not None else None
        so += H * n
        r["idx"], r["k_out"], r["v_out"] = [], [], []
        for h in range(H):
            c, o = int(counts[b * H + h]), int(offsets[b * H + h])
            r["idx"].append(idx[o:o + c].astype(np.int64))
            r["k_out"].append(k_out[o:o + c])
            r["v_out"].append(v_out[o:o + c])
        out.append(r)
    return out


def assert_scores_close(gpu, ora, what):
    gpu = np.asarray(gpu, np.float64)
    ora = np.asarray(ora, np.float64)
    tol = RTOL * np.abs(ora) + ATOL_FRAC * np.max(np.abs(ora))
    err = np.abs(gpu - ora)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err / np.maximum(tol, 1e-300)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} scores outside tolerance; worst at {i}: "
                             f"gpu {gpu[i]!r} oracle {ora[i]!r}")
    return float(np.max(err / np.maximum(np.abs(ora), 1e-30) * (np.abs(ora) > ATOL_FRAC * np.max(np.abs(ora)))))


def kth_key(scores, forced, budget):
    """Score of the budget-th entry in (forced first, score desc, index asc) order, or
    None when the budget is filled by forced entries."""
    nf = int(forced.sum())
    if budget <= nf:
        return None
    free = np.sort(scores[~forced])[::-1]
    return free[budget - nf - 1]


def near(x, t):
    return t is not None and abs(x - t) <= SEL_RTOL * abs(t)


def check_selection_near_ties(gpu_idx, ora_idx, forced, n, budget, thresholds, what):
    """GPU and oracle kept sets may differ only by entries whose oracle score is within
    SEL_RTOL of one of the thresholds [(scores, T), ...]."""
    g = np.asarray(gpu_idx)
    assert len(g) == budget, f"{what}: kept {len(g)} != budget {budget}"
    assert np.all(np.diff(g) > 0), f"{what}: indices not strictly ascending"
    assert g.size == 0 or (g[0] >= 0 and g[-1] < n), f"{what}: index out of range"
    assert set(np.flatnonzero(forced).tolist()) <= set(g.tolist()), f"{what}: forced entry dropped"
    diff = set(g.tolist()) ^ set(np.asarray(ora_idx).tolist())
    for i in diff:
        assert any(near(s[i], t) for s, t in thresholds), (
            f"{what}: entry {i} differs and is not a near-tie: " + ", ".join(f"{s[i]!r} vs T {t!r}" for s, t in thresholds))
    return len(diff)


def check_topk_property(scores, kept, forced, budget, what):
    """Kept set equals the top-`budget` of `scores` (forced first, score desc, ties by
    index asc) — checked on the GPU's own scores, by comparison of keys."""
    n = len(scores)
    kept = np.asarray(kept)
    assert len(kept) == budget, what
    mask = np.zeros(n, bool)
    mask[kept] = True
    assert np.all(mask[forced]), what
    free_k = mask & ~forced
    free_d = ~mask & ~forced
    if free_k.any() and free_d.any():
        lo = scores[free_k].min()
        hi = scores[free_d].max()
        assert lo >= hi, f"{what}: dropped score {hi!r} above kept {lo!r}"
        if lo == hi:  # ties at the threshold: kept ones come first by index
            tk = np.flatnonzero(free_k & (scores == lo))
            td = np.flatnonzero(free_d & (scores == lo))
            assert tk.max() < td.min(), f"{what}: tie order violated"


def topk_mask(scores, forced, budget):
    """Mask of the top-`budget` entries of `scores` (forced first, score desc, index asc).
    Used only to check the GPU's selection against the GPU's own scores."""
    n = len(scores)
    key = np.where(forced, np.inf, np.asarray(scores, np.float64))
    order = np.lexsort((np.arange(n), -key))
    m = np.zeros(n, bool)
    m[order[:budget]] = True
    return m
