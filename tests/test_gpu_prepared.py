"""Value-norm weights prepared once per model (kvsel_prepare_w_o) against W_O passed to
every call: the same kernels read the same W_h (or Gram matrix), so every score, kept
index and compacted row must be bit-identical ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을
최적화하기", §3.4 Algorithm 1 and App. D.4: W_h is a function of the model's weights alone)."""
import numpy as np
import pytest

from kv_cache_eviction_window_gb300 import datagen
from tests import gpu_harness as GH

pytestmark = pytest.mark.gpu


def _run(wl, inp, prepared, **override):
    import torch

    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding as B

    n = inp["n_ctx"][0]
    p = B.params_from_workload(wl, n_ctx=n, w_o_prepared=prepared, **override)
    q = GH.torch_bf16(inp["q"])
    k, v = GH.torch_bf16(inp["k"][0]), GH.torch_bf16(inp["v"][0])
    kv = B.make_kv_contiguous(k, v)
    w = GH.torch_bf16(inp["w_o"])
    buf = B.LayerBuffers(p)
    if prepared:
        p0 = B.params_from_workload(wl, n_ctx=n, **override)
        ws0 = torch.zeros(B.kvsel_workspace_size(p0) // 4 + 64, dtype=torch.int32, device="cuda")
        B.kvsel_workspace_init(ws0)
        wp = torch.empty(B.kvsel_prepared_w_o_size(p) // 2 + 128, dtype=torch.int16, device="cuda")
        B.kvsel_prepare_w_o(p, w, wp, ws0)
        w = wp
    B.kvsel_run_layer(p, q, kv, w, buf.s_attn, buf.s_val, buf.idx, buf.counts, buf.offsets, buf.k_out, buf.v_out,
                      buf.ws)
    torch.cuda.synchronize()
    assert B.kvsel_get_device_status(buf.ws) == 0
    return {k_: getattr(buf, k_).cpu() for k_ in ("s_attn", "s_val", "idx", "counts", "offsets", "k_out", "v_out")}


def _same_bits(a, b):
    import torch

    for key in a:
        x = a[key].contiguous().view(torch.uint8).numpy()
        y = b[key].contiguous().view(torch.uint8).numpy()
        np.testing.assert_array_equal(x, y, err_msg=key)


@pytest.mark.parametrize("override", [dict(), dict(value_norm="l2"), dict(wo_mode="per_head")])
def test_prepared_weights_are_bit_identical(override):
    wl = datagen.WORKLOADS[2].replace(layers=1)
    inp = datagen.make_layer(wl, 3, n_ctx=2085)
    _same_bits(_run(wl, inp, False, **override), _run(wl, inp, True, **override))


@pytest.mark.parametrize("concurrent", [False, True])
def test_prepared_weights_full_size_layer(concurrent):
    """The benchmark's 32K layer: prepared and per-call weights give the same outputs, bit
    for bit (the per-call path is compared with the full oracle in test_gpu_parity), alone
    and as an overlapping call (the benchmark's configuration)."""
    wl = datagen.WORKLOADS[2]
    inp = datagen.make_layer(wl, 0)
    _same_bits(_run(wl, inp, False, concurrent=concurrent), _run(wl, inp, True, concurrent=concurrent))


def test_prepared_sizes_and_rejections():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding as B

    wl = datagen.WORKLOADS[2]
    p = B.params_from_workload(wl)
    assert B.kvsel_prepared_w_o_size(p) == wl.h_kv * wl.d_model * 128 * 2
    assert B.kvsel_prepared_w_o_size(B.params_from_workload(wl, value_norm="l2")) == wl.h_kv * 2 * 128 * 128 * 2
    # plain scoring has no value-norm weights
    with pytest.raises(B.KvselError):
        B.kvsel_prepared_w_o_size(B.params_from_workload(wl, value_aware=False))
    # a buffer one element short is refused before any launch
    w = torch.zeros(16, dtype=torch.int16, device="cuda")
    short = torch.empty(B.kvsel_prepared_w_o_size(p) // 2 - 128, dtype=torch.int16, device="cuda")
    with pytest.raises(B.KvselError) as e:
        B.kvsel_prepare_w_o(p, w, short)
    assert e.value.code == B.KVSEL_EINVAL
