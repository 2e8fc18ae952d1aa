"""The exchange between ranks for one budget per layer when the layer's KV heads are
spread over ranks.

The per-layer budget ("KVzip: Query-Agnostic KV Cache Compression with Context
Reconstruction", §4.2; "CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", §3.4 Algorithm 2,
line 1) ranks every entry of a layer together, so a rank that holds only some heads of the
layer cannot choose its entries alone.  This module is the agreement between the ranks,
the one exchange the path needs when a layer is sharded; choosing the entries stays where
the keys live (per-head floors need no exchange, since a head lives on one rank):

* the layer threshold key T (the budget-th largest order-preserving 32-bit key over every
  rank's entries, floor picks counted as the largest key): radix passes over 8-bit
  digits, each pass one all-reduce (sum) of the ranks' 256-bin histograms of the keys
  still in play (``layer_threshold``);
* ties at T, broken as on one device (flat index h*n + i ascending): one all-reduce of
  every head's count of keys equal to T gives each head the number of its ties that are
  taken (``ties_taken``).

Only histograms and per-head counts cross ranks, never scores or indices.  On one GB300
the library never splits a layer (each device runs whole layers: replicas), so nothing on
the device path calls this module; the tests drive it with CPU process groups, with the
local histograms and the final extraction computed on the host, and compare the result
with a single-device selection.
"""
from __future__ import annotations

from typing import Callable, Sequence, Tuple

import numpy as np


class Comm:
    """The one collective the exchange uses (an element-wise sum over ranks) on a
    torch.distributed process group; with none initialised, a single rank."""

    def __init__(self, group=None):
        self.group = group
        self.dist = None
        try:
            import torch.distributed as dist

            if dist.is_available() and dist.is_initialized():
                self.dist = dist
        except ImportError:  # pragma: no cover - torch is always present here
            pass

    def sum(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.int64)
        if self.dist is None:
            return x
        import torch

        t = torch.from_numpy(x.copy())
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM, group=self.group)
        return t.numpy()


def layer_threshold(local_hist: Callable[[int, int, int], np.ndarray], budget: int, comm: Comm) -> Tuple[int, int]:
    """(T, krem): the budget-th largest key over every rank's keys, and how many keys equal
    to T the layer takes.  local_hist(prefix, mask, shift) returns this rank's 256-bin
    histogram of the digit (key >> shift) & 255 over its keys with (key & mask) == prefix.
    Every rank gets the same answer.  Raises ValueError when the budget exceeds the
    layer's entries."""
    if budget <= 0:
        return 0xFFFFFFFF, 0
    prefix, mask, krem = 0, 0, int(budget)
    for shift in (24, 16, 8, 0):
        h = comm.sum(local_hist(prefix, mask, shift))
        above = 0
        for d in range(255, -1, -1):   # the largest digits first
            if above < krem <= above + int(h[d]):
                prefix |= d << shift
                krem -= above
                break
            above += int(h[d])
        else:
            raise ValueError("budget above the number of entries")
        mask |= 0xFF << shift
    return prefix, krem


def ties_taken(eq_local: Sequence[int], heads: Sequence[int], n_heads: int, krem: int, comm: Comm) -> np.ndarray:
    """Per local head, how many of its keys equal to T are taken: ties go to the lowest
    flat indices first, so to heads in id order.  eq_local[j]: the count of keys equal to T
    in head heads[j] of this rank."""
    eq = np.zeros(n_heads, dtype=np.int64)
    for j, hid in enumerate(heads):
        eq[hid] = int(eq_local[j])
    eq = comm.sum(eq)   # each head is counted on its one rank: the sum gathers them
    out = np.zeros(len(heads), dtype=np.int64)
    for j, hid in enumerate(heads):
        before = int(eq[:hid].sum())
        out[j] = max(0, min(int(eq[hid]), int(krem) - before))
    return out
