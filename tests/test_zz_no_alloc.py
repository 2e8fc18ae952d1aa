"""kvsel_score_noalloc against kvsel_score.

The no-allocation entry point serves callers that cannot call cudaMalloc (a process whose
device memory belongs to a preallocated arena such as a serving engine's KV-cache pool,
or a path that must not synchronise the device).  It scores with the library's built-in
scratch buffer instead of a caller workspace; its results must match the workspace entry
point's within the score tolerance of the other GPU tests, on two calls in a row that
follow a call on a different request (the shared buffer keeps the previous call's
contents), for contiguous and paged caches; errors found on the device must be readable
through kvsel_get_device_status(NULL); and requests larger than the buffer must be refused
before any launch.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

from kv_cache_eviction_window_gb300 import datagen
from tests import gpu_harness as GH

pytestmark = pytest.mark.gpu


def _inputs(B, wl, seed, n, paged):
    import torch

    inp = datagen.make_layer(wl, seed, n_ctx=n)
    p = B.params_from_workload(wl, n_ctx=n)
    q = GH.torch_bf16(inp["q"])
    if paged:
        pg = inp["paged"]
        k, v = GH.torch_bf16(pg["k_pool"]), GH.torch_bf16(pg["v_pool"])
        table = torch.from_numpy(pg["block_table"][:1]).cuda()
        kv = B.make_kv_paged(k, v, table)
        keep = (k, v, table)
    else:
        k, v = GH.torch_bf16(inp["k"][0]), GH.torch_bf16(inp["v"][0])
        kv = B.make_kv_contiguous(k, v)
        keep = (k, v)
    w = GH.torch_bf16(inp["w_o"])
    return p, q, kv, w, keep


def _scores_with_workspace(B, p, q, kv, w):
    import torch

    n_scores, _, _ = B.kvsel_output_size(p)
    ws = torch.empty(B.kvsel_workspace_size(p) // 4 + 64, dtype=torch.int32, device="cuda")
    B.kvsel_workspace_init(ws)
    a = torch.empty(n_scores, dtype=torch.float32, device="cuda")
    s = torch.empty(n_scores, dtype=torch.float32, device="cuda")
    B.kvsel_score(p, q, kv, w, a, s, ws)
    torch.cuda.synchronize()
    assert B.kvsel_get_device_status(ws) == 0
    return a.cpu().numpy(), s.cpu().numpy()


def _scores_noalloc(B, p, q, kv, w):
    import torch

    n_scores, _, _ = B.kvsel_output_size(p)
    a = torch.full((n_scores,), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.full((n_scores,), float("nan"), dtype=torch.float32, device="cuda")
    B.kvsel_score_noalloc(p, q, kv, w, a, s)
    torch.cuda.synchronize()
    return a.cpu().numpy(), s.cpu().numpy(), B.kvsel_get_device_status(None)


@pytest.mark.parametrize("paged", [False, True])
def test_noalloc_matches_workspace_entry_point_twice(paged):
    """The built-in buffer first holds another request's scratch (a longer context, other
    inputs), then the checked request runs twice in a row; both calls must match
    kvsel_score with a workspace, so nothing left in the buffer leaks into a result."""
    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding as B

    wl = datagen.WORKLOADS[4 if paged else 2].replace(layers=1, batch=1)
    # a different, larger request fills the buffer with unrelated partials and scores
    other = _inputs(B, wl, 11, 7000, paged)
    assert B.kvsel_workspace_size(other[0]) <= B.NOALLOC_SCRATCH_BYTES
    _, _, st = _scores_noalloc(B, *other[:4])
    assert st == 0
    p, q, kv, w, keep = _inputs(B, wl, 5, 3000, paged)
    assert B.kvsel_workspace_size(p) <= B.NOALLOC_SCRATCH_BYTES
    ref_a, ref_v = _scores_with_workspace(B, p, q, kv, w)
    for call in range(2):
        a, s, st = _scores_noalloc(B, p, q, kv, w)
        assert st == 0, f"device status {st} after no-alloc call {call}"
        GH.assert_scores_close(a, ref_a, f"s_attn, no-alloc call {call}")
        GH.assert_scores_close(s, ref_v, f"s_val, no-alloc call {call}")


def test_noalloc_reports_device_errors_through_the_status_word():
    """A bounded wait that runs out inside a no-alloc call (wait budget of 1 cycle) is seen
    through kvsel_get_device_status(NULL); the next call starts from a clear status word
    and scores correctly."""
    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding as B

    wl = datagen.WORKLOADS[2].replace(layers=1)
    p, q, kv, w, keep = _inputs(B, wl, 5, 3000, False)
    ref_a, ref_v = _scores_with_workspace(B, p, q, kv, w)
    p1 = B.params_from_workload(wl, n_ctx=3000, wait_cycles=1)
    _, _, st = _scores_noalloc(B, p1, q, kv, w)
    assert st == B.KVSEL_ETIMEOUT
    assert B.kvsel_get_device_status(None) == 0   # read and cleared
    a, s, st = _scores_noalloc(B, p, q, kv, w)
    assert st == 0
    GH.assert_scores_close(a, ref_a, "s_attn after a timed-out call")
    GH.assert_scores_close(s, ref_v, "s_val after a timed-out call")


def test_noalloc_refuses_requests_beyond_its_buffer():
    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding as B

    # a 16-request ragged batch of up to 64K tokens needs well over the 16 MiB buffer
    wl = datagen.WORKLOADS[4]
    lens = datagen.context_lengths(wl)
    p = B.params_from_workload(wl, n_ctx_per_req=lens)
    assert B.kvsel_workspace_size(p) > B.NOALLOC_SCRATCH_BYTES
    kv = B.kvsel_kv()
    with pytest.raises(B.KvselError) as e:
        B.kvsel_score_noalloc(p, 16, kv, 16, 16, 16, 0)
    assert e.value.code == B.KVSEL_EWORKSPACE
    np.testing.assert_equal(e.value.code, -4)
