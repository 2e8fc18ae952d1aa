"""Output perturbation of a kept set on the GPU against the fp64 oracle ("CriticalKV: 출력
섭동 관점에서 KV 캐시 축출을 최적화하기", Definition 3.1, Theorems 3.2, 3.3, C.1, Table 9).

The kept sets come from the oracle's own selection, or from a seeded random draw; the
GPU computes the actual perturbation and both bounds per window row of every query head.
Tolerance: relative 1e-3 (the score tolerance of the other parity tests) with an absolute
floor of 1e-5 of the largest value of each quantity per head.  The error of the actual
perturbation is bounded by u * theta, theta the Theorem 3.3 bound of the same row (the sum
of |c_i| ||v'_i||_1 over the keys), u about 2^-17 for the bf16 high and low parts of the
weights plus the fp32 accumulation over the keys; theta is at most about 6x the actual
value on these layers, far inside 1e-3.
"""
import numpy as np
import pytest

from kv_cache_eviction_window_gb300 import datagen
from tests import gpu_harness as GH

pytestmark = pytest.mark.gpu

RTOL = 1e-3
AFLOOR = 1e-5


def run_gpu_perturbation(wl, inp, kept, paged=False):
    import torch
    from kv_cache_eviction_window_gb300 import binding as B
    from tests.test_gpu_anchor import _kv_for

    lens = inp["n_ctx"]
    p = B.params_from_workload(wl, n_ctx_per_req=lens if len(lens) > 1 else None, n_ctx=lens[0])
    q = GH.torch_bf16(inp["q"])
    kv, keep = _kv_for(wl, inp, paged)
    w = GH.torch_bf16(inp["w_o"])
    flat = np.concatenate([np.asarray(kk, np.int32) for req in kept for kk in req]).astype(np.int32)
    cnt = np.array([len(kk) for req in kept for kk in req], np.int32)
    off = np.concatenate([[0], np.cumsum(cnt)[:-1]]).astype(np.int64)
    idx = torch.from_numpy(flat if len(flat) else np.zeros(1, np.int32)).cuda()
    counts = torch.from_numpy(cnt).cuda()
    offsets = torch.from_numpy(off).cuda()
    H, G, W = wl.h_kv, wl.group, wl.window
    out = torch.full((len(lens), H, 3, G, W), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(B.kvsel_perturbation_workspace_size(p) // 4 + 64, dtype=torch.int32, device="cuda")
    B.kvsel_workspace_init(ws)
    B.kvsel_perturbation(p, q, kv, w, idx, counts, offsets, out, ws)
    torch.cuda.synchronize()
    status = B.kvsel_get_device_status(ws)
    del keep
    assert status == 0, f"device status {status}"
    return out.cpu().numpy().astype(np.float64)


def compare(gpu, ora, heads=None):
    for b, o in enumerate(ora):
        for h in (range(o.shape[0]) if heads is None else heads):
            for k, name in enumerate(("actual", "bound", "relaxed bound")):
                g = gpu[b, h, k]
                w = o[h, k]
                tol = RTOL * np.abs(w) + AFLOOR * np.abs(w).max()
                bad = np.abs(g - w) > tol
                assert not bad.any(), (f"req {b} head {h} {name}: {bad.sum()} rows off; worst gpu "
                                       f"{g[bad][0]!r} oracle {w[bad][0]!r}")


def kept_from_oracle(wl, inp, value_aware):
    from oracle import kvsel_oracle as O

    r = O.run_workload_layer(wl.replace(value_aware=value_aware), inp, compact_out=False)
    return [x["idx"] for x in r]


@pytest.mark.parametrize("value_aware", [False, True])
def test_perturbation_small_both_selections(value_aware):
    from oracle import perturb_oracle as PO

    wl = datagen.WORKLOADS[2].replace(layers=1, h_kv=2, d_model=1024)
    inp = datagen.make_layer(wl, 0, n_ctx=1000)
    kept = kept_from_oracle(wl, inp, value_aware)
    gpu = run_gpu_perturbation(wl, inp, kept)
    ora = PO.run_perturbation_layer(inp["q"], inp["k"], inp["v"], inp["w_o"], kept, group=wl.group)
    compare(gpu, ora)
    # the bound chain holds on the GPU's numbers too
    assert (gpu[0, :, 0] <= gpu[0, :, 1] * (1 + 1e-3) + 1e-6).all()
    assert (gpu[0, :, 1] <= gpu[0, :, 2] * (1 + 1e-3) + 1e-6).all()


def test_perturbation_ragged_paged_random_kept_sets():
    from oracle import perturb_oracle as PO

    wl = datagen.WORKLOADS[4].replace(batch=3, n_min=300, n_ctx=1500, d_model=512)
    inp = datagen.make_layer(wl, 0)
    rng = np.random.default_rng(5)
    kept = []
    for n in inp["n_ctx"]:
        req = []
        for h in range(wl.h_kv):
            free = rng.choice(n - 32, size=(n - 32) // 3, replace=False)
            req.append(np.union1d(free, np.arange(n - 32, n)))
        kept.append(req)
    gpu = run_gpu_perturbation(wl, inp, kept, paged=True)
    ora = PO.run_perturbation_layer(inp["q"], inp["k"], inp["v"], inp["w_o"], kept, group=wl.group)
    compare(gpu, ora)


def test_perturbation_keep_all_is_zero():
    wl = datagen.WORKLOADS[2].replace(layers=1, h_kv=2, d_model=512)
    inp = datagen.make_layer(wl, 0, n_ctx=700)
    kept = [[np.arange(700) for _ in range(2)]]
    gpu = run_gpu_perturbation(wl, inp, kept)
    for k, name in enumerate(("actual", "bound", "relaxed bound")):
        assert np.abs(gpu[:, :, k]).max() == 0.0, name


def test_perturbation_full_size_one_head():
    # the 32K Llama-3.1-8B layer (D = 4096) with the oracle's value-aware kept set; the
    # oracle checks head 3
    from oracle import kvsel_oracle as O
    from oracle import perturb_oracle as PO

    wl = datagen.WORKLOADS[2].replace(layers=1)
    inp = datagen.make_layer(wl, 0)
    r = O.run_workload_layer(wl, inp, compact_out=False, heads=[3])[0]
    n = wl.n_ctx
    kept = [[r["idx"][h] if h == 3 else np.arange(n - 4096, n) for h in range(wl.h_kv)]]
    gpu = run_gpu_perturbation(wl, inp, kept)
    ora = PO.run_perturbation_layer(inp["q"], inp["k"], inp["v"], inp["w_o"], kept, group=wl.group, heads=[3])
    compare(gpu, ora, heads=[3])


def test_perturbation_rejects_unsupported_shapes():
    # 448 window rows per head (Qwen2.5-7B: G = 7, W = 64) exceed one 128-row tile
    from kv_cache_eviction_window_gb300 import binding as B

    p = B.params_from_workload(datagen.WORKLOADS[3].replace(d_model=3584))
    with pytest.raises(B.KvselError) as e:
        B.kvsel_perturbation_workspace_size(p)
    assert e.value.code == B.KVSEL_EUNSUPPORTED
    # query-agnostic scoring has no window rows
    p = B.params_from_workload(datagen.WORKLOADS[5].replace(d_model=8192))
    with pytest.raises(B.KvselError) as e:
        B.kvsel_perturbation_workspace_size(p)
    assert e.value.code == B.KVSEL_EUNSUPPORTED
