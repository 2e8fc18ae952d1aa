"""kvsel_partition against the oracle: the kept set and its complement.

"VestigeKV: The NoPE-MLA KV Cache Carries Its Own Eviction Signal in a Vestigial Branch",
§4.1: eviction moves rows to an archive and deletes nothing, so the kept side and the
archived side partition every segment's positions.  The evicted index lists must equal
the oracle's complement of the kept list (bit-exact, ascending), the archived and kept
rows must be the cache's rows bit for bit, and the per-segment counts and offsets must
follow from the kept counts.
"""
import numpy as np
import pytest

from kv_cache_eviction_window_gb300 import datagen
from oracle import kvsel_oracle as O
from tests import gpu_harness as GH

pytestmark = pytest.mark.gpu


def _lib():
    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding as B

    return B


def _run(wl, inp, paged, **override):
    """kvsel_run_layer, then kvsel_partition of its kept set; numpy outputs per request."""
    import torch

    B = _lib()
    lens = inp["n_ctx"]
    bsz = len(lens)
    p = B.params_from_workload(wl, n_ctx_per_req=lens if bsz > 1 else None, n_ctx=lens[0], **override)
    q = GH.torch_bf16(inp["q"])
    if paged:
        pg = inp["paged"]
        kt, vt = GH.torch_bf16(pg["k_pool"]), GH.torch_bf16(pg["v_pool"])
        table = torch.from_numpy(pg["block_table"]).cuda()
        kv = B.make_kv_paged(kt, vt, table)
    else:
        H, d = wl.h_kv, wl.head_dim
        nmax = max(lens)
        kc = np.zeros((bsz, H, nmax, d), np.uint16)
        vc = np.zeros((bsz, H, nmax, d), np.uint16)
        for b in range(bsz):
            kc[b, :, :lens[b]] = inp["k"][b]
            vc[b, :, :lens[b]] = inp["v"][b]
        kt, vt = GH.torch_bf16(kc), GH.torch_bf16(vc)
        kv = B.make_kv_contiguous(kt, vt)
    w_o = GH.torch_bf16(inp["w_o"]) if p.value_aware else None
    buf = B.LayerBuffers(p)
    B.kvsel_run_layer(p, q, kv, w_o, buf.s_attn, buf.s_val, buf.idx, buf.counts, buf.offsets, buf.k_out, buf.v_out,
                      buf.ws)
    n_ev = buf.n_scores - buf.n_kept
    ev_idx = torch.full((max(n_ev, 1),), -7, dtype=torch.int32, device="cuda")
    ev_counts = torch.full((buf.n_seg,), -7, dtype=torch.int32, device="cuda")
    ev_offsets = torch.full((buf.n_seg,), -7, dtype=torch.int64, device="cuda")
    k_ev = torch.zeros((max(n_ev, 1), 128), dtype=torch.bfloat16, device="cuda")
    v_ev = torch.zeros_like(k_ev)
    k_kept = torch.zeros_like(buf.k_out)
    v_kept = torch.zeros_like(buf.v_out)
    B.kvsel_partition(p, kv, buf.idx, buf.counts, buf.offsets, ev_idx, ev_counts, ev_offsets, k_ev, v_ev, k_kept,
                      v_kept, buf.ws)
    torch.cuda.synchronize()
    status = B.kvsel_get_device_status(buf.ws)

    def u16(t):
        return t.cpu().view(torch.int16).numpy().view(np.uint16)

    return dict(p=p, status=status, idx=buf.idx.cpu().numpy(), counts=buf.counts.cpu().numpy(),
                offsets=buf.offsets.cpu().numpy(), ev_idx=ev_idx.cpu().numpy(), ev_counts=ev_counts.cpu().numpy(),
                ev_offsets=ev_offsets.cpu().numpy(), k_ev=u16(k_ev), v_ev=u16(v_ev), k_kept=u16(k_kept),
                v_kept=u16(v_kept), k_out=u16(buf.k_out), v_out=u16(buf.v_out), n_ev=n_ev)


def _check(wl, inp, r, heads=None):
    H = wl.h_kv
    assert r["status"] == 0, f"device status {r['status']}"
    np.testing.assert_array_equal(r["k_kept"], r["k_out"])   # one pass writes what kvsel_compact wrote
    np.testing.assert_array_equal(r["v_kept"], r["v_out"])
    ev_total = 0
    for b, n in enumerate(inp["n_ctx"]):
        for h in range(H):
            s = b * H + h
            c, o = int(r["counts"][s]), int(r["offsets"][s])
            kept = r["idx"][o:o + c].astype(np.int64)
            ora_kept, ora_ev = O.partition(n, kept)
            np.testing.assert_array_equal(ora_kept, kept)
            assert int(r["ev_counts"][s]) == n - c
            assert int(r["ev_offsets"][s]) == ev_total, (b, h)
            eo = ev_total
            ev_total += n - c
            if heads is not None and h not in heads:
                continue
            np.testing.assert_array_equal(r["ev_idx"][eo:eo + n - c], ora_ev, err_msg=f"ev_idx b{b} h{h}")
            np.testing.assert_array_equal(r["k_ev"][eo:eo + n - c], O.archive(inp["k"][b][h], kept))
            np.testing.assert_array_equal(r["v_ev"][eo:eo + n - c], O.archive(inp["v"][b][h], kept))
    assert ev_total == r["n_ev"]


def test_partition_c2_full_layer():
    """The 32K Llama-3.1-8B layer (value-aware two-stage selection): 8 heads of 32768
    positions, 19661 archived per head; every evicted index and row is checked."""
    wl = datagen.WORKLOADS[2]
    inp = datagen.make_layer(wl, 0)
    _check(wl, inp, _run(wl, inp, paged=False))


def test_partition_ragged_paged_batch():
    """Ragged requests in a paged cache (block 16, shuffled block table), per-head budget."""
    wl = datagen.WORKLOADS[4].replace(batch=5, n_min=1500, n_ctx=9000, d_model=512)
    inp = datagen.make_layer(wl, 0)
    _check(wl, inp, _run(wl, inp, paged=True))


def test_partition_per_layer_budget():
    """A budget per layer (KVzip §4.2): counts differ between heads, and so do the
    archived counts and offsets."""
    wl = datagen.WORKLOADS[3]
    inp = datagen.make_layer(wl, 0, n_ctx=5000)
    r = _run(wl, inp, paged=False)
    assert len(set(r["counts"].tolist())) > 1
    _check(wl, inp, r)


def test_partition_rejects_inconsistent_kept_lists():
    """An unsorted kept list and a count beyond the segment are skipped and flagged
    (KVSEL_EDEVICE); nothing outside the outputs is written (the guard rows stay)."""
    import torch

    B = _lib()
    wl = datagen.WORKLOADS[1].replace(h_kv=2)
    n = 640
    inp = datagen.make_layer(wl, 0, n_ctx=n)
    p = B.params_from_workload(wl, n_ctx=n)
    kt, vt = GH.torch_bf16(inp["k"][0]), GH.torch_bf16(inp["v"][0])
    kv = B.make_kv_contiguous(kt, vt)
    n_scores, n_kept, n_seg = B.kvsel_output_size(p)
    bud = n_kept // 2
    good = np.arange(0, n, n // bud)[:bud].astype(np.int32)
    bad = good.copy()
    bad[[3, 40]] = bad[[40, 3]]   # not ascending
    idx = torch.from_numpy(np.concatenate([good, bad])).cuda()
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")
    n_ev = n_scores - n_kept
    guard = 64

    def call(counts):
        ev_idx = torch.full((n_ev + guard,), -7, dtype=torch.int32, device="cuda")
        k_ev = torch.full((n_ev + guard, 128), 3.0, dtype=torch.bfloat16, device="cuda")
        v_ev = torch.full((n_ev + guard, 128), 3.0, dtype=torch.bfloat16, device="cuda")
        evc = torch.zeros(n_seg, dtype=torch.int32, device="cuda")
        evo = torch.zeros(n_seg, dtype=torch.int64, device="cuda")
        cnt = torch.tensor(counts, dtype=torch.int32, device="cuda")
        off = torch.tensor([0, counts[0]], dtype=torch.int64, device="cuda")
        B.kvsel_partition(p, kv, idx, cnt, off, ev_idx, evc, evo, k_ev, v_ev, None, None, ws)
        torch.cuda.synchronize()
        return B.kvsel_get_device_status(ws), ev_idx.cpu().numpy(), k_ev.float().cpu().numpy(), evc.cpu().numpy()

    st, ev_idx, k_ev, evc = call([bud, bud])
    assert st == B.KVSEL_EDEVICE
    # head 0 (sorted list) is partitioned exactly; nothing lands past the outputs
    _, ora_ev = O.partition(n, good)
    np.testing.assert_array_equal(ev_idx[:n - bud], ora_ev)
    assert np.all(ev_idx[n_ev:] == -7) and np.all(k_ev[n_ev:] == 3.0)
    assert evc.tolist() == [n - bud, n - bud]
    st, ev_idx, k_ev, evc = call([bud, n + 5])   # a count beyond the segment
    assert st == B.KVSEL_EDEVICE
    assert evc.tolist() == [n - bud, 0]
    assert np.all(ev_idx[n_ev:] == -7) and np.all(k_ev[n_ev:] == 3.0)
