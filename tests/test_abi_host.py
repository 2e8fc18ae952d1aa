"""Host-side checks of the C ABI (no GPU): the library builds and loads, exports every
function include/kvsel.h declares, sizes its outputs as the budgets say, and rejects
bad arguments before any CUDA work."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding

    binding.load()
    return binding


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvsel.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvsel_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(B):
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert set(names) <= set(B.EXPORTS)


def test_version_and_errors(B):
    assert "sm_103a" in B.kvsel_version()
    for code in range(0, -8, -1):
        assert B.kvsel_strerror(code) and "unknown" not in B.kvsel_strerror(code)


def test_struct_layout_matches_header(B):
    # compile-time sizes of the C structs (gcc, same ABI as the binding's ctypes structs)
    import subprocess
    import tempfile

    src = '#include <stdio.h>\n#include <stddef.h>\n#include "kvsel.h"\nint main(){printf("%zu %zu %zu %zu %zu %zu %zu\\n",' \
          'sizeof(kvsel_params), sizeof(kvsel_kv), offsetof(kvsel_params, budget_ratio),' \
          'offsetof(kvsel_kv, block_table), offsetof(kvsel_params, wait_cycles),' \
          'offsetof(kvsel_params, sm_budget), offsetof(kvsel_params, concurrent));return 0;}\n'
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "s.c")
        open(c, "w").write(src)
        exe = os.path.join(d, "s")
        subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe])
        out = subprocess.check_output([exe]).decode().split()
    want = [ctypes.sizeof(B.kvsel_params), ctypes.sizeof(B.kvsel_kv), B.kvsel_params.budget_ratio.offset,
            B.kvsel_kv.block_table.offset, B.kvsel_params.wait_cycles.offset, B.kvsel_params.sm_budget.offset,
            B.kvsel_params.concurrent.offset]
    assert [int(x) for x in out] == want


@pytest.mark.parametrize("cid", [1, 2, 3, 4])
def test_output_sizes_follow_budgets(B, cid):
    from kv_cache_eviction_window_gb300 import datagen

    wl = datagen.WORKLOADS[cid]
    lens = datagen.context_lengths(wl)
    p = B.params_from_workload(wl, n_ctx_per_req=lens if wl.batch > 1 else None)
    n_scores, n_kept, n_seg = B.kvsel_output_size(p)
    assert n_scores == wl.h_kv * sum(lens)
    assert n_seg == wl.h_kv * len(lens)
    if wl.budget_mode == "head":
        want = sum(wl.h_kv * math.floor(wl.budget_ratio * n) for n in lens)
    else:
        want = sum(math.floor(wl.budget_ratio * n * wl.h_kv) for n in lens)
    assert n_kept == want


def _p(B, **kw):
    base = dict(h_kv=8, group=4, n_ctx=4096, window=32, budget_ratio=0.2)
    base.update(kw)
    return B.make_params(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), -3),
    (dict(h_kv=0), -1),
    (dict(pool="max", pool_kernel=4), -1),
    (dict(budget_ratio=0.005), -2),            # 20 slots < 36 forced entries
    (dict(budget_ratio=1.5), -1),
    (dict(window=0, causal=True, reduce="max"), -3),     # query-agnostic scoring is non-causal
    (dict(window=0, causal=False, reduce="mean"), -3),   # ... and takes the max over queries
    (dict(window=0, causal=False, reduce="max", value_aware=True, d_model=4096), -3),
    (dict(group=3, window=10), -3),             # 30 window rows: not a multiple of 32
    (dict(window=8192), -1),                    # window longer than the context
    (dict(sm_budget=-1), -1),                   # a negative SM budget
    (dict(value_aware=True, d_model=4096, budget_mode="anchor"), -3),
    (dict(value_aware=True, d_model=100), -3),
    (dict(value_aware=True, d_model=4096, value_norm="l2", wo_mode="per_head"), -3),   # Gram needs one W_h
    (dict(budget_mode="layer", budget_ratio=0.1, floor_ratio=0.2), -2),
])
def test_invalid_parameters(B, kw, code):
    p = _p(B, **kw)
    with pytest.raises(B.KvselError) as e:
        B.kvsel_output_size(p)
    assert e.value.code == code


def test_select_rejects_null_pointers(B):
    p = _p(B)
    lib = B.load()
    rc = lib.kvsel_select(ctypes.byref(p), None, None, None, None, None, None, 0, None)
    assert rc == B.KVSEL_EINVAL


def test_empty_request_is_a_no_op(B):
    p = _p(B, n_ctx=0, n_recent=0, n_sink=0, window=32)
    assert B.kvsel_output_size(p) == (0, 0, 8)


def test_query_agnostic_sizes(B):
    p = _p(B, window=0, causal=False, reduce="max", pool="none", n_recent=0,
           budget_mode="layer", budget_ratio=0.3, n_ctx=32768)
    n_scores, n_kept, n_seg = B.kvsel_output_size(p)
    assert (n_scores, n_kept, n_seg) == (8 * 32768, math.floor(0.3 * 32768 * 8), 8)


def test_ex2_probe_rejects_null_and_misaligned_arguments(B):
    import bench

    f = bench.load_ex2_probe()
    a, b = ctypes.c_double(), ctypes.c_double()
    assert f(None, 4096, ctypes.byref(a), ctypes.byref(b)) == -1
    assert f(16, 4096, None, ctypes.byref(b)) == -1
    assert f(24, 4096, ctypes.byref(a), ctypes.byref(b)) == -1


def test_probe_is_not_part_of_the_library(B):
    lib = ctypes.CDLL(B.LIB_PATH)
    assert not hasattr(lib, "kvsel_probe_ex2_rate")
    assert not hasattr(lib, "kvsel_set_wait_limit")   # the wait budget is a per-call parameter
