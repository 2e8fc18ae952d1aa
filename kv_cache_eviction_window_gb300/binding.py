"""ctypes binding of libkvsel (include/kvsel.h): same entry-point names, argument
marshalling only.  Device buffers are torch CUDA tensors (torch is the allocator and
the stream provider); every step of the computation runs in libkvsel's kernels.

There is no fallback: if the shared library is missing or fails to load, every call
raises ``KvselUnavailable``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkvsel.so")

KVSEL_OK = 0
KVSEL_EINVAL = -1
KVSEL_EBUDGET = -2
KVSEL_EUNSUPPORTED = -3
KVSEL_EWORKSPACE = -4
KVSEL_ECUDA = -5
KVSEL_ETIMEOUT = -6
KVSEL_EDEVICE = -7

REDUCE = {"sum": 0, "mean": 1, "max": 2, "max_logit": 3}
POOL = {"none": 0, "max": 1, "avg": 2}
BUDGET = {"head": 0, "layer": 1, "anchor": 2}
WO_MODE = {"group_sum": 0, "per_head": 1}
VALUE_NORM = {"l1": 0, "l2": 1}
LAYOUT_CONTIGUOUS, LAYOUT_PAGED = 0, 1
MAX_BATCH = 128

EXPORTS = ("kvsel_workspace_size", "kvsel_output_size", "kvsel_workspace_init", "kvsel_score",
           "kvsel_select", "kvsel_compact", "kvsel_partition", "kvsel_run_layer", "kvsel_get_device_status",
           "kvsel_set_stage_events", "kvsel_strerror", "kvsel_version",
           "kvsel_score_noalloc", "kvsel_launch_count", "kvsel_head_scores", "kvsel_anchor_project",
           "kvsel_run_anchors", "kvsel_perturbation_workspace_size", "kvsel_perturbation",
           "kvsel_query_agnostic_split", "kvsel_prepared_w_o_size", "kvsel_prepare_w_o")
NOALLOC_SCRATCH_BYTES = 16 << 20
STAGES = ("rowstats", "keysum", "wbar", "vnorm", "finalize", "select", "compact", "project", "perturb")


class KvselUnavailable(RuntimeError):
    pass


class KvselError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


class kvsel_params(ctypes.Structure):
    _fields_ = [
        ("h_kv", ctypes.c_int32), ("group", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("d_model", ctypes.c_int32), ("n_ctx", ctypes.c_int32), ("window", ctypes.c_int32),
        ("q_chunk", ctypes.c_int32), ("causal", ctypes.c_int32), ("scale", ctypes.c_float),
        ("reduce", ctypes.c_int32), ("pool", ctypes.c_int32), ("pool_kernel", ctypes.c_int32),
        ("value_aware", ctypes.c_int32), ("wo_mode", ctypes.c_int32), ("eps", ctypes.c_float),
        ("alpha", ctypes.c_float), ("n_sink", ctypes.c_int32), ("n_recent", ctypes.c_int32),
        ("budget_mode", ctypes.c_int32), ("budget_ratio", ctypes.c_double),
        ("floor_ratio", ctypes.c_double), ("batch", ctypes.c_int32),
        ("n_ctx_per_req", ctypes.POINTER(ctypes.c_int32)), ("value_norm", ctypes.c_int32),
        ("w_o_prepared", ctypes.c_int32), ("wait_cycles", ctypes.c_uint64), ("sm_budget", ctypes.c_int32),
        ("concurrent", ctypes.c_int32),
    ]


class kvsel_kv(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("layout", ctypes.c_int32),
        ("stride_req", ctypes.c_int64), ("stride_head", ctypes.c_int64), ("stride_tok", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("block_size", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
    ]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libkvsel.so (built by __graft_entry__.build()); raise if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise KvselUnavailable(f"libkvsel.so not built ({p}); run __graft_entry__.build()")
    try:
        lib = ctypes.CDLL(p)
    except OSError as e:  # pragma: no cover - depends on the machine
        raise KvselUnavailable(f"cannot load {p}: {e}") from e
    P, K = ctypes.POINTER(kvsel_params), ctypes.POINTER(kvsel_kv)
    vp, sz, i64p = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int64)
    sig = {
        "kvsel_workspace_size": ([P, ctypes.POINTER(sz)], ctypes.c_int),
        "kvsel_output_size": ([P, i64p, i64p, i64p], ctypes.c_int),
        "kvsel_workspace_init": ([vp, sz, vp], ctypes.c_int),
        "kvsel_score": ([P, vp, K, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "kvsel_select": ([P, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "kvsel_compact": ([P, K, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "kvsel_partition": ([P, K] + [vp] * 11 + [sz, vp], ctypes.c_int),
        "kvsel_run_layer": ([P, vp, K, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "kvsel_get_device_status": ([vp, vp, ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
        "kvsel_set_stage_events": ([ctypes.c_void_p], None),
        "kvsel_score_noalloc": ([P, vp, K, vp, vp, vp, vp], ctypes.c_int),
        "kvsel_strerror": ([ctypes.c_int], ctypes.c_char_p),
        "kvsel_version": ([], ctypes.c_char_p),
        "kvsel_launch_count": ([], ctypes.c_uint64),
        "kvsel_head_scores": ([P, vp, vp, vp], ctypes.c_int),
        "kvsel_prepared_w_o_size": ([P, ctypes.POINTER(sz)], ctypes.c_int),
        "kvsel_prepare_w_o": ([P, vp, vp, sz, vp, sz, vp], ctypes.c_int),
        "kvsel_query_agnostic_split": ([P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)],
                                       ctypes.c_int),
        "kvsel_anchor_project": ([P, K] + [vp] * 10 + [sz, vp], ctypes.c_int),
        "kvsel_run_anchors": ([P, vp, K] + [vp] * 12 + [sz, vp], ctypes.c_int),
        "kvsel_perturbation_workspace_size": ([P, ctypes.POINTER(sz)], ctypes.c_int),
        "kvsel_perturbation": ([P, vp, K, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    if path is None:
        _lib = lib
    return lib


# ------------------------------------------------------------------------------ helpers
def make_params(*, h_kv: int, group: int, n_ctx: int, window: int, head_dim: int = 128,
                d_model: int = 0, q_chunk: int = 0, causal: bool = True, scale: float = 0.0,
                reduce: str = "mean", pool: str = "max", pool_kernel: int = 7,
                value_aware: bool = False, wo_mode: str = "group_sum", eps: float = 1e-4,
                alpha: float = 0.5, n_sink: int = 4, n_recent: int = 32,
                budget_mode: str = "head", budget_ratio: float = 0.2, floor_ratio: float = 0.0,
                n_ctx_per_req: Optional[Sequence[int]] = None, value_norm: str = "l1",
                wait_cycles: int = 0, w_o_prepared: bool = False, sm_budget: int = 0,
                concurrent: bool = False) -> kvsel_params:
    p = kvsel_params()
    p.h_kv, p.group, p.head_dim, p.d_model = h_kv, group, head_dim, d_model
    p.n_ctx, p.window, p.q_chunk, p.causal = n_ctx, window, q_chunk, int(bool(causal))
    p.scale = scale
    p.reduce, p.pool, p.pool_kernel = REDUCE[reduce], POOL[pool], pool_kernel
    p.value_aware, p.wo_mode, p.eps, p.alpha = int(bool(value_aware)), WO_MODE[wo_mode], eps, alpha
    p.n_sink, p.n_recent = n_sink, n_recent
    p.budget_mode, p.budget_ratio, p.floor_ratio = BUDGET[budget_mode], budget_ratio, floor_ratio
    p.value_norm = VALUE_NORM[value_norm]
    p.wait_cycles = int(wait_cycles)
    p.sm_budget = int(sm_budget)
    p.concurrent = int(bool(concurrent))
    p.w_o_prepared = int(bool(w_o_prepared))
    if n_ctx_per_req is not None:
        arr = (ctypes.c_int32 * len(n_ctx_per_req))(*[int(x) for x in n_ctx_per_req])
        p._n_arr = arr  # keep alive
        p.n_ctx_per_req = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
        p.batch = len(n_ctx_per_req)
    else:
        p.batch = 1
    return p


def params_from_workload(wl, n_ctx_per_req: Optional[Sequence[int]] = None, **override) -> kvsel_params:
    kw = dict(h_kv=wl.h_kv, group=wl.group, n_ctx=wl.n_ctx, window=wl.window, head_dim=wl.head_dim,
              d_model=wl.d_model if wl.value_aware else 0, q_chunk=wl.q_chunk, causal=wl.causal,
              reduce=wl.reduce, pool=wl.pool, pool_kernel=wl.pool_kernel, value_aware=wl.value_aware,
              eps=wl.eps, alpha=wl.alpha, n_sink=wl.n_sink, n_recent=wl.n_recent,
              budget_mode=wl.budget_mode, budget_ratio=wl.budget_ratio, floor_ratio=wl.floor_ratio,
              n_ctx_per_req=n_ctx_per_req, value_norm=wl.value_norm)
    kw.update(override)
    return make_params(**kw)


def make_kv_contiguous(k, v, *, stride_req: int = 0) -> kvsel_kv:
    """K/V tensors [H][n][d] (one request) or [B][H][n][d] (bf16, CUDA)."""
    kv = kvsel_kv()
    kv.k, kv.v = _ptr(k), _ptr(v)
    kv.layout = LAYOUT_CONTIGUOUS
    kv.stride_tok = k.stride(-2)
    kv.stride_head = k.stride(-3)
    kv.stride_req = k.stride(-4) if k.dim() == 4 else stride_req
    return kv


def make_kv_paged(k_pool, v_pool, block_table) -> kvsel_kv:
    """Pools [num_blocks][block][H][d] bf16 and block_table [B][max_blocks] int32 (CUDA)."""
    kv = kvsel_kv()
    kv.k, kv.v = _ptr(k_pool), _ptr(v_pool)
    kv.layout = LAYOUT_PAGED
    kv.block_table = _ptr(block_table)
    kv.block_size = k_pool.shape[1]
    kv.max_blocks = block_table.shape[1]
    kv.num_blocks = k_pool.shape[0]
    return kv


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> None:
    if rc != KVSEL_OK:
        raise KvselError(rc, where)


# ------------------------------------------------------------------------------ the ABI
def strerror(code: int) -> str:
    try:
        return load().kvsel_strerror(code).decode()
    except KvselUnavailable:
        return f"error {code}"


def kvsel_version() -> str:
    return load().kvsel_version().decode()


def kvsel_strerror(code: int) -> str:
    return load().kvsel_strerror(code).decode()


def kvsel_launch_count() -> int:
    return int(load().kvsel_launch_count())


def kvsel_prepared_w_o_size(params) -> int:
    out = ctypes.c_size_t()
    _check(load().kvsel_prepared_w_o_size(ctypes.byref(params), ctypes.byref(out)), "kvsel_prepared_w_o_size")
    return out.value


def kvsel_prepare_w_o(params, w_o, w_prep, ws=None, stream=None) -> None:
    """The value-norm weights of W_O (W_h, or its Gram matrix for the L2 norm) into w_prep,
    once per model; scoring calls with w_o_prepared=True then take w_prep as their w_o."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().kvsel_prepare_w_o(ctypes.byref(params), _ptr(w_o), _ptr(w_prep),
                                    w_prep.numel() * w_prep.element_size(), _ptr(ws), nbytes, _stream(stream)),
           "kvsel_prepare_w_o")


def kvsel_query_agnostic_split(params) -> tuple:
    """(key blocks per head, query-row slices per key block) of query-agnostic scoring."""
    kb, rs = ctypes.c_int32(), ctypes.c_int32()
    _check(load().kvsel_query_agnostic_split(ctypes.byref(params), ctypes.byref(kb), ctypes.byref(rs)),
           "kvsel_query_agnostic_split")
    return kb.value, rs.value


def kvsel_head_scores(params, scores, head_out, stream=None) -> None:
    """head_out[b*h_kv + h] = max over the sequence of request b, head h of `scores`."""
    _check(load().kvsel_head_scores(ctypes.byref(params), _ptr(scores), _ptr(head_out), _stream(stream)),
           "kvsel_head_scores")


def kvsel_set_stage_events(events) -> None:
    """events: None, or a ctypes array of 2*len(STAGES) cudaEvent_t handles (kept alive
    by the caller while set)."""
    load().kvsel_set_stage_events(None if events is None else ctypes.cast(events, ctypes.c_void_p))


def kvsel_workspace_size(params: kvsel_params) -> int:
    out = ctypes.c_size_t()
    _check(load().kvsel_workspace_size(ctypes.byref(params), ctypes.byref(out)), "kvsel_workspace_size")
    return out.value


def kvsel_output_size(params: kvsel_params):
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(load().kvsel_output_size(ctypes.byref(params), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
           "kvsel_output_size")
    return a.value, b.value, c.value


def kvsel_workspace_init(ws, stream=None) -> None:
    _check(load().kvsel_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_workspace_init")


def kvsel_score(params, q, kv: kvsel_kv, w_o, s_attn, s_val, ws, stream=None) -> None:
    _check(load().kvsel_score(ctypes.byref(params), _ptr(q), ctypes.byref(kv), _ptr(w_o), _ptr(s_attn),
                              _ptr(s_val), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_score")


def kvsel_score_noalloc(params, q, kv: kvsel_kv, w_o, s_attn, s_val, stream=None) -> None:
    """kvsel_score with the library's built-in scratch buffer instead of a workspace, for
    callers that cannot allocate device memory (see include/kvsel.h)."""
    _check(load().kvsel_score_noalloc(ctypes.byref(params), _ptr(q), ctypes.byref(kv), _ptr(w_o), _ptr(s_attn),
                                      _ptr(s_val), _stream(stream)), "kvsel_score_noalloc")


def kvsel_select(params, s_attn, s_val, idx, counts, offsets, ws=None, stream=None) -> None:
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().kvsel_select(ctypes.byref(params), _ptr(s_attn), _ptr(s_val), _ptr(idx), _ptr(counts),
                               _ptr(offsets), _ptr(ws), nbytes, _stream(stream)), "kvsel_select")


def kvsel_compact(params, kv: kvsel_kv, idx, counts, offsets, k_out, v_out, ws=None, stream=None) -> None:
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().kvsel_compact(ctypes.byref(params), ctypes.byref(kv), _ptr(idx), _ptr(counts), _ptr(offsets),
                                _ptr(k_out), _ptr(v_out), _ptr(ws), nbytes, _stream(stream)), "kvsel_compact")


def kvsel_partition(params, kv: kvsel_kv, idx, counts, offsets, ev_idx, ev_counts, ev_offsets, k_ev, v_ev,
                    k_kept=None, v_kept=None, ws=None, stream=None) -> None:
    """Kept set and its complement: evicted positions and the evicted (and optionally the
    kept) K/V rows, bit-exact."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().kvsel_partition(ctypes.byref(params), ctypes.byref(kv), _ptr(idx), _ptr(counts), _ptr(offsets),
                                  _ptr(ev_idx), _ptr(ev_counts), _ptr(ev_offsets), _ptr(k_ev), _ptr(v_ev),
                                  _ptr(k_kept), _ptr(v_kept), _ptr(ws), nbytes, _stream(stream)), "kvsel_partition")


def kvsel_run_layer(params, q, kv: kvsel_kv, w_o, s_attn, s_val, idx, counts, offsets, k_out, v_out, ws,
                    stream=None) -> None:
    _check(load().kvsel_run_layer(ctypes.byref(params), _ptr(q), ctypes.byref(kv), _ptr(w_o), _ptr(s_attn),
                                  _ptr(s_val), _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(k_out),
                                  _ptr(v_out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_run_layer")


def kvsel_anchor_project(params, kv: kvsel_kv, anchor_k, anchor_v, idx, counts, offsets, slot_k, gamma_k,
                         slot_v, gamma_v, ws, stream=None) -> None:
    _check(load().kvsel_anchor_project(ctypes.byref(params), ctypes.byref(kv), _ptr(anchor_k), _ptr(anchor_v),
                                       _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(slot_k), _ptr(gamma_k),
                                       _ptr(slot_v), _ptr(gamma_v), _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream)), "kvsel_anchor_project")


def kvsel_run_anchors(params, q, kv: kvsel_kv, rand_keys, s_attn, idx, counts, offsets, anchor_k, anchor_v,
                      slot_k, gamma_k, slot_v, gamma_v, ws, stream=None) -> None:
    _check(load().kvsel_run_anchors(ctypes.byref(params), _ptr(q), ctypes.byref(kv), _ptr(rand_keys),
                                    _ptr(s_attn), _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(anchor_k),
                                    _ptr(anchor_v), _ptr(slot_k), _ptr(gamma_k), _ptr(slot_v), _ptr(gamma_v),
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "kvsel_run_anchors")


def kvsel_perturbation_workspace_size(params: kvsel_params) -> int:
    out = ctypes.c_size_t()
    _check(load().kvsel_perturbation_workspace_size(ctypes.byref(params), ctypes.byref(out)),
           "kvsel_perturbation_workspace_size")
    return out.value


def kvsel_perturbation(params, q, kv: kvsel_kv, w_o, idx, counts, offsets, out, ws, stream=None) -> None:
    _check(load().kvsel_perturbation(ctypes.byref(params), _ptr(q), ctypes.byref(kv), _ptr(w_o), _ptr(idx),
                                     _ptr(counts), _ptr(offsets), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)), "kvsel_perturbation")


def kvsel_get_device_status(ws, stream=None) -> int:
    """Read and clear the status word of workspace `ws`, or with ws=None the one of the
    built-in buffer that kvsel_score_noalloc uses on the current device."""
    st = ctypes.c_int()
    _check(load().kvsel_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(st)), "kvsel_get_device_status")
    return st.value


# ------------------------------------------------------------------------------ buffers
class LayerBuffers:
    """Device outputs and workspace for one layer call (torch allocations)."""

    def __init__(self, params: kvsel_params, device="cuda"):
        import torch

        n_scores, n_kept, n_seg = kvsel_output_size(params)
        ws_bytes = kvsel_workspace_size(params)
        self.s_attn = torch.empty(max(n_scores, 1), dtype=torch.float32, device=device)
        self.s_val = torch.empty(max(n_scores, 1), dtype=torch.float32, device=device) if params.value_aware else None
        self.idx = torch.empty(max(n_kept, 1), dtype=torch.int32, device=device)
        self.counts = torch.empty(max(n_seg, 1), dtype=torch.int32, device=device)
        self.offsets = torch.empty(max(n_seg, 1), dtype=torch.int64, device=device)
        self.k_out = torch.empty((max(n_kept, 1), params.head_dim), dtype=torch.bfloat16, device=device)
        self.v_out = torch.empty((max(n_kept, 1), params.head_dim), dtype=torch.bfloat16, device=device)
        self.ws = torch.empty(max(ws_bytes, 256) // 4 + 64, dtype=torch.int32, device=device)
        if params.budget_mode == BUDGET["anchor"]:
            # anchors: per-position slot and gamma for K and V (k_out / v_out hold the anchors)
            self.slot_k = torch.empty(max(n_scores, 1), dtype=torch.int32, device=device)
            self.slot_v = torch.empty(max(n_scores, 1), dtype=torch.int32, device=device)
            self.gamma_k = torch.empty(max(n_scores, 1), dtype=torch.float32, device=device)
            self.gamma_v = torch.empty(max(n_scores, 1), dtype=torch.float32, device=device)
        kvsel_workspace_init(self.ws)
        self.n_scores, self.n_kept, self.n_seg = n_scores, n_kept, n_seg
