"""kvsel_score_noalloc against kvsel_score.

The no-allocation entry point serves callers that cannot call cudaMalloc (a process whose
device memory belongs to a preallocated arena such as a serving engine's KV-cache pool,
or a path that must not synchronise the device).  It scores with the library's built-in
scratch buffer instead of a caller workspace; its results must match the workspace entry
point's within the score tolerance of the other GPU tests, on two calls in a row (the
shared buffer keeps the previous call's contents), and requests larger than the buffer
must be refused before any launch.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

from kv_cache_eviction_window_gb300 import datagen
from tests import gpu_harness as GH

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding as B

    wl = datagen.WORKLOADS[2].replace(layers=1)
    inp = datagen.make_layer(wl, 5, n_ctx=3000)
    p = B.params_from_workload(wl, n_ctx=3000)
    q = GH.torch_bf16(inp["q"])
    k = GH.torch_bf16(inp["k"][0])
    v = GH.torch_bf16(inp["v"][0])
    w = GH.torch_bf16(inp["w_o"])
    kv = B.make_kv_contiguous(k, v)
    n_scores, _, _ = B.kvsel_output_size(p)
    assert B.kvsel_workspace_size(p) <= B.NOALLOC_SCRATCH_BYTES

    ws = torch.empty(B.kvsel_workspace_size(p) // 4 + 64, dtype=torch.int32, device="cuda")
    B.kvsel_workspace_init(ws)
    ref_a = torch.empty(n_scores, dtype=torch.float32, device="cuda")
    ref_v = torch.empty(n_scores, dtype=torch.float32, device="cuda")
    B.kvsel_score(p, q, kv, w, ref_a, ref_v, ws)
    torch.cuda.synchronize()
    assert B.kvsel_get_device_status(ws) == 0
    ref_a, ref_v = ref_a.cpu().numpy(), ref_v.cpu().numpy()

    for call in range(2):
        a = torch.full((n_scores,), float("nan"), dtype=torch.float32, device="cuda")
        s = torch.full((n_scores,), float("nan"), dtype=torch.float32, device="cuda")
        B.kvsel_score_noalloc(p, q, kv, w, a, s)
        torch.cuda.synchronize()
        GH.assert_scores_close(a.cpu().numpy(), ref_a, f"s_attn, no-alloc call {call}")
        GH.assert_scores_close(s.cpu().numpy(), ref_v, f"s_val, no-alloc call {call}")


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
