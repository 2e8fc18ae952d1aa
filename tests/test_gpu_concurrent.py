"""Calls running at the same time on several streams (kvsel_params.concurrent = 1).

Independent layers may be issued over several streams, each call with its own workspace
and outputs.  With concurrent = 1 a call uses only kernels that make progress whatever
else is resident (the two scoring passes as two launches, no cooperative grid barrier),
so overlapping calls cannot wait on each other.  These tests check that path against the
oracle for the window-row counts the single cooperative launch would otherwise take, and
that layers issued over three streams give, bit for bit, what the same calls give one
after the other (CriticalKV §3.4, Algorithm 2; KVzip §4.2)."""
import numpy as np
import pytest

from kv_cache_eviction_window_gb300 import datagen
from oracle import kvsel_oracle as O
from tests import gpu_harness as GH
from tests.test_gpu_parity import _check_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding

    binding.load()
    yield


@pytest.mark.parametrize("group,window,value_aware,budget", [(4, 32, True, 76), (4, 32, False, 76),
                                                             (2, 32, True, 76), (8, 32, False, 76),
                                                             (4, 64, True, 76), (4, 32, True, 24),
                                                             (4, 32, False, 24)])
def test_two_launch_scoring_matches_the_oracle(group, window, value_aware, budget):
    # an SM budget of 24 for 8 heads selects on 2-CTA clusters (4 per head would exceed it)
    wl = datagen.WORKLOADS[2].replace(layers=1, group=group, window=window, value_aware=value_aware)
    inp = datagen.make_layer(wl, 21, n_ctx=3001)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp, concurrent=True, sm_budget=budget)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("reduce,causal,group,window", [("sum", True, 4, 24), ("max", True, 5, 32),
                                                         ("mean", False, 1, 32), ("max", False, 8, 40),
                                                         ("sum", True, 2, 48)])
def test_two_launch_reductions_and_ragged_window_rows(reduce, causal, group, window):
    # window rows R = group * window: 96, 160, 32, 320 (one pass-2 accumulator) and 96, so
    # that pass 2's last block of rows is a lone 32-row block and the causal tail
    # crosses the row blocks
    wl = datagen.WORKLOADS[1].replace(reduce=reduce, causal=causal, group=group, window=window, h_kv=2,
                                      pool="max", pool_kernel=5)
    inp = datagen.make_layer(wl, 5, n_ctx=2345)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp, concurrent=True, sm_budget=40)
    _check_layer(wl, inp, gpu, ora)


@pytest.mark.parametrize("cid,n,kw", [(3, 3333, dict()), (3, 2500, dict(value_aware=True, d_model=1024)),
                                      (4, None, dict(batch=4, n_min=300, n_ctx=1400))])
def test_concurrent_selection_per_layer_and_batched(cid, n, kw):
    # overlapping calls select on 4-CTA clusters: per-layer budgets with floors (one
    # segment per layer), the value-aware two-stage selection under a per-layer budget,
    # and the ragged paged batch, each against the oracle
    wl = datagen.WORKLOADS[cid].replace(**kw)
    inp = datagen.make_layer(wl, 9, n_ctx=n) if n else datagen.make_layer(wl, 9)
    ora = O.run_workload_layer(wl, inp)
    gpu = GH.run_gpu_layer(wl, inp, concurrent=True, sm_budget=76)
    _check_layer(wl, inp, gpu, ora)


def test_layers_over_three_streams_match_one_stream():
    import torch

    from kv_cache_eviction_window_gb300 import binding as B

    wl = datagen.WORKLOADS[2].replace(layers=1)
    n = 6000
    nl, ns = 6, 3
    dev = torch.device("cuda", 0)
    p = B.params_from_workload(wl, n_ctx=n, concurrent=True, sm_budget=76)
    layers = []
    for i in range(nl):
        x = datagen.make_layer(wl, 40 + i, n_ctx=n)
        q = GH.torch_bf16(x["q"])
        k, v = GH.torch_bf16(x["k"][0]), GH.torch_bf16(x["v"][0])
        w = GH.torch_bf16(x["w_o"])
        layers.append((q, k, v, B.make_kv_contiguous(k, v), w))

    def run(streams):
        outs = []
        bufs = [B.LayerBuffers(p, device=dev) for _ in range(nl)]
        ws = [torch.zeros(B.kvsel_workspace_size(p) // 4 + 64, dtype=torch.int32, device=dev) for _ in streams]
        for x in ws:
            B.kvsel_workspace_init(x)
        torch.cuda.synchronize()
        for i, (q, _, _, kv, w) in enumerate(layers):
            j = i % len(streams)
            b = bufs[i]
            B.kvsel_run_layer(p, q, kv, w, b.s_attn, b.s_val, b.idx, b.counts, b.offsets, b.k_out, b.v_out, ws[j],
                              streams[j])
        torch.cuda.synchronize()
        for x in ws:
            assert B.kvsel_get_device_status(x) == 0
        for b in bufs:
            outs.append({k_: getattr(b, k_).cpu() for k_ in ("s_attn", "s_val", "idx", "counts", "offsets", "k_out",
                                                             "v_out")})
        return outs

    one = run([torch.cuda.Stream()])
    many = run([torch.cuda.Stream() for _ in range(ns)])
    for i in range(nl):
        for key in one[i]:
            np.testing.assert_array_equal(one[i][key].contiguous().view(torch.uint8).numpy(),
                                          many[i][key].contiguous().view(torch.uint8).numpy(), err_msg=f"{i} {key}")
