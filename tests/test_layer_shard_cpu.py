"""The exchange for one budget per layer across ranks (layer_shard) on two gloo ranks.

A layer's heads are split over two CPU processes; each rank builds its heads' keys (floor
picks at the largest key), the ranks agree on the layer threshold through summed
histograms and on the ties through summed per-head counts, and each rank keeps its
entries.  The union must equal the oracle's single-device per-layer selection (KVzip §4.2
top over all heads, per-head floors, ties by flat index), including ties planted across
heads on different ranks."""
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _keys(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return np.where(u >> 31, ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def _case(seed):
    rng = np.random.default_rng(seed)
    H, n = 4, 300
    s = rng.random((H, n)).astype(np.float32) * np.float32(1e-3)
    # ties across heads on both ranks, at about the layer threshold and elsewhere
    s[0, 10:20] = s[1, 40:50] = s[2, 5:9] = s[3, 100:130] = np.float32(6.0e-4)
    s[1, 200:210] = s[2, 210:220] = np.float32(2.5e-4)
    fm = np.zeros((H, n), bool)
    fm[:, :4] = True
    fm[:, -8:] = True
    return s, fm, 340 + 17 * seed, 40


def _local_select(s, fm, heads, n_heads, budget, floor, group=None):
    """One rank's part: keys of its heads, the exchange, then its kept entries."""
    from kv_cache_eviction_window_gb300 import layer_shard as LS

    comm = LS.Comm(group)
    keys = []
    for hid in heads:
        k = _keys(s[hid])
        k[fm[hid]] = 0xFFFFFFFF
        f = min(len(k), max(floor, int(fm[hid].sum())))
        free = np.flatnonzero(~fm[hid])
        order = free[np.lexsort((free, -s[hid][free].astype(np.float64)))]
        k[order[:f - int(fm[hid].sum())]] = 0xFFFFFFFF
        keys.append(k)
    flat = np.concatenate(keys)

    def hist(prefix, mask, shift):
        sel = flat[(flat & np.uint32(mask)) == np.uint32(prefix)]
        return np.bincount(((sel >> np.uint32(shift)) & np.uint32(255)).astype(np.int64), minlength=256)

    T, krem = LS.layer_threshold(hist, budget, comm)
    take = LS.ties_taken([int((k == np.uint32(T)).sum()) for k in keys], heads, n_heads, krem, comm)
    out = {}
    for j, hid in enumerate(heads):
        ties = np.flatnonzero(keys[j] == np.uint32(T))[:take[j]]
        out[hid] = np.union1d(np.flatnonzero(keys[j] > np.uint32(T)), ties)
    return out


def _worker(rank, world, port, seed, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    s, fm, budget, floor = _case(seed)
    heads = [h for h in range(s.shape[0]) if h % world == rank]   # heads 0, 2 | 1, 3
    out = _local_select(s, fm, heads, s.shape[0], budget, floor)
    q.put((rank, {h: v.tolist() for h, v in out.items()}))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_two_ranks_match_the_single_device_selection(seed):
    import multiprocessing as mp

    from oracle import kvsel_oracle as O

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, seed, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(2):
        rank, res = q.get(timeout=180)
        got.update({int(h): v for h, v in res.items()})
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    s, fm, budget, floor = _case(seed)
    want = O.select_per_layer(s.astype(np.float64), budget, fm, floor)
    assert sum(len(v) for v in got.values()) == budget
    for h in range(s.shape[0]):
        assert got[h] == want[h].tolist(), f"head {h}"


def test_one_rank_without_a_process_group():
    """The same exchange with no process group initialised: a single rank holding every head."""
    from oracle import kvsel_oracle as O

    s, fm, budget, floor = _case(3)
    got = _local_select(s, fm, list(range(s.shape[0])), s.shape[0], budget, floor)
    want = O.select_per_layer(s.astype(np.float64), budget, fm, floor)
    for h in range(s.shape[0]):
        np.testing.assert_array_equal(got[h], want[h])


def test_budget_above_the_layer_is_refused():
    from kv_cache_eviction_window_gb300 import layer_shard as LS

    with pytest.raises(ValueError):
        LS.layer_threshold(lambda p, m, sh: np.zeros(256, np.int64), 5, LS.Comm())
