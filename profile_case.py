"""Run a few layers of one workload through kvsel_run_layer, for profilers (ncu).

    python profile_case.py --workload 2 --layers 2 --steps 2
    python profile_case.py --workload 2 --value-norm l2
    python profile_case.py --workload 6      # AnchorKV anchors
    python profile_case.py --workload 2 --perturb   # + output perturbation
    python profile_case.py --workload 5 --n-ctx 8192  # query-agnostic, smaller n
    python profile_case.py --workload 2 --plain --partition   # + kept/evicted partition
    python profile_case.py --workload 2 --plain --concurrent --sm-budget 76   # two-launch scoring
    python profile_case.py --workload 2 --plain --layers 8 --graph-streams 8 --concurrent --sm-budget 76

With --graph-streams S the layers are issued round-robin over S streams (one workspace
each) and captured as one CUDA graph; after --steps warm-up replays, one more replay runs
between cudaProfilerStart and cudaProfilerStop, for `ncu --profile-from-start off
--graph-profiling graph`, which measures the whole replay (all layers, overlapped) as one
result.

The inputs are the same seeded synthetic tensors as the benchmark (each layer distinct,
larger than L2 for the 32K stack), so per-launch counters taken here scale to the
benchmark's full stack.  Prints per-stage CUDA-event times; it is not a benchmark line.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--layers", type=int, default=2)
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--plain", action="store_true", help="value_aware=0")
    ap.add_argument("--value-norm", default=None, choices=["l1", "l2"], help="value-aware norm override")
    ap.add_argument("--perturb", action="store_true", help="also run kvsel_perturbation on each layer's kept set")
    ap.add_argument("--n-ctx", type=int, default=None, help="context length override (a smaller case of the shape)")
    ap.add_argument("--partition", action="store_true", help="also run kvsel_partition on each layer's kept set")
    ap.add_argument("--concurrent", action="store_true", help="kvsel_params.concurrent = 1 (two-launch scoring)")
    ap.add_argument("--sm-budget", type=int, default=0, help="kvsel_params.sm_budget")
    ap.add_argument("--graph-streams", type=int, default=0,
                    help="issue the layers over this many streams as one CUDA graph (see above)")
    args = ap.parse_args()
    import numpy as np
    import torch

    import __graft_entry__

    __graft_entry__.build()
    from kv_cache_eviction_window_gb300 import binding as B
    from kv_cache_eviction_window_gb300 import datagen

    wl = datagen.WORKLOADS[args.workload]
    if args.plain:
        wl = wl.replace(value_aware=False)
    if args.value_norm:
        wl = wl.replace(value_norm=args.value_norm)
    if args.n_ctx:
        wl = wl.replace(n_ctx=args.n_ctx)
    anchors = wl.budget_mode == "anchor"
    dev = torch.device("cuda", 0)

    def to_dev(u16):
        return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(dev)

    layers = []
    x_w = {}   # W_O per layer for the perturbation (also when the scoring is not value-aware)
    for layer in range(args.layers):
        x = datagen.make_layer(wl, layer)
        lens = x["n_ctx"]
        p = B.params_from_workload(wl, n_ctx_per_req=lens if len(lens) > 1 else None, n_ctx=lens[0],
                                   concurrent=args.concurrent, sm_budget=args.sm_budget)
        if wl.paged:
            pg = x["paged"]
            kt, vt = to_dev(pg["k_pool"]), to_dev(pg["v_pool"])
            table = torch.from_numpy(pg["block_table"]).to(dev)
            kv = B.make_kv_paged(kt, vt, table)
            keep = (kt, vt, table)
        else:
            kt, vt = to_dev(np.stack(x["k"])), to_dev(np.stack(x["v"]))
            kv = B.make_kv_contiguous(kt, vt)
            keep = (kt, vt)
        q = to_dev(x["q"])
        w = to_dev(x["w_o"]) if wl.value_aware else None
        if anchors:   # the random keys of the anchor draw ride in the weight slot
            w = torch.from_numpy(np.concatenate([r.reshape(-1) for r in x["rand"]])).to(dev)
        buf = B.LayerBuffers(p, device=dev)
        x_w[id(buf)] = to_dev(x["w_o"]) if x["w_o"] is not None else None
        layers.append((p, q, kv, w, buf, keep))
    if args.graph_streams > 0:
        return run_graph(args, B, layers, dev)
    nst = len(B.STAGES)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * nst)]
    for e in ev:
        e.record()
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * (2 * nst))(*[e.cuda_event for e in ev])
    tot = [0.0] * nst
    cnt = 0
    for _ in range(args.steps):
        for (p, q, kv, w, b, _k) in layers:
            B.kvsel_set_stage_events(arr)
            if anchors:
                B.kvsel_run_anchors(p, q, kv, w, b.s_attn, b.idx, b.counts, b.offsets, b.k_out, b.v_out, b.slot_k,
                                    b.gamma_k, b.slot_v, b.gamma_v, b.ws)
            else:
                B.kvsel_run_layer(p, q, kv, w, b.s_attn, b.s_val, b.idx, b.counts, b.offsets, b.k_out, b.v_out,
                                  b.ws)
            if args.partition:
                if not hasattr(b, "ev_idx"):
                    n_ev = max(b.n_scores - b.n_kept, 1)
                    b.ev_idx = torch.empty(n_ev, dtype=torch.int32, device=dev)
                    b.ev_counts = torch.empty(b.n_seg, dtype=torch.int32, device=dev)
                    b.ev_offsets = torch.empty(b.n_seg, dtype=torch.int64, device=dev)
                    b.k_ev = torch.empty((n_ev, 128), dtype=torch.bfloat16, device=dev)
                    b.v_ev = torch.empty((n_ev, 128), dtype=torch.bfloat16, device=dev)
                B.kvsel_partition(p, kv, b.idx, b.counts, b.offsets, b.ev_idx, b.ev_counts, b.ev_offsets, b.k_ev,
                                  b.v_ev, b.k_out, b.v_out, b.ws)
            if args.perturb:
                if not hasattr(b, "pt_out"):
                    b.pt_out = torch.empty((1, wl.h_kv, 3, wl.group, wl.window), dtype=torch.float32, device=dev)
                    b.pt_ws = torch.zeros(B.kvsel_perturbation_workspace_size(p) // 4 + 64, dtype=torch.int32,
                                          device=dev)
                    B.kvsel_workspace_init(b.pt_ws)
                B.kvsel_perturbation(p, q, kv, x_w[id(b)], b.idx, b.counts, b.offsets, b.pt_out, b.pt_ws)
            B.kvsel_set_stage_events(None)
            torch.cuda.synchronize()
            for i in range(nst):
                try:
                    tot[i] += ev[2 * i].elapsed_time(ev[2 * i + 1])
                except RuntimeError:
                    pass
            cnt += 1
    st = B.kvsel_get_device_status(layers[0][4].ws)
    print(f"workload {wl.name} (value_aware={wl.value_aware}), {args.layers} layers x {args.steps} steps, "
          f"device status {st}")
    for i, name in enumerate(B.STAGES):
        print(f"  {name:9s} {tot[i] / cnt * 1e3:9.2f} us/layer (event-timed, includes launch gaps)")
    return 0 if st == 0 else 1


def run_graph(args, B, layers, dev):
    """The layers over S streams as one CUDA graph; the last replay is the profiled one."""
    import torch

    S = args.graph_streams
    p0 = layers[0][0]
    wss = [torch.zeros(B.kvsel_workspace_size(p0) // 4 + 64, dtype=torch.int32, device=dev) for _ in range(S)]
    for x in wss:
        B.kvsel_workspace_init(x)
    ss = [torch.cuda.Stream() for _ in range(S)]

    def issue():
        for i, (p, q, kv, w, b, _k) in enumerate(layers):
            B.kvsel_run_layer(p, q, kv, w, b.s_attn, b.s_val, b.idx, b.counts, b.offsets, b.k_out, b.v_out,
                              wss[i % S], ss[i % S])

    issue()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=ss[0]):
        for x in ss[1:]:
            x.wait_stream(ss[0])
        issue()
        for x in ss[1:]:
            ss[0].wait_stream(x)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(max(args.steps, 1)):
        t0.record()
        g.replay()
        t1.record()
        torch.cuda.synchronize()
        times.append(t0.elapsed_time(t1))
    torch.cuda.profiler.start()
    g.replay()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    st = [B.kvsel_get_device_status(x) for x in wss]
    print(f"{len(layers)} layers over {S} streams as one graph: best replay {min(times) * 1e3 / len(layers):.2f} "
          f"us/layer, device status {st}")
    return 0 if not any(st) else 1


if __name__ == "__main__":
    sys.exit(main())
