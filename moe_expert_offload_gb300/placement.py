"""Static expert placements for moe_cache_place (host logic, no device work).

The pages compare FreeToken's shared LRU against the placement policies of two
edge engines, replayed on the same routing traces (FreeToken summary "Key
results" and "core method": KTransformers fixes its "hot" experts when the
model loads, llama.cpp assigns whole layers to a device; reader Figure 4(b)).
These two functions choose those sets; the cache then runs with
MOE_POLICY_STATIC, so the set never changes and every miss is executed from
the bank.
"""
from __future__ import annotations

import numpy as np


def hot_placement(trace: np.ndarray, num_experts: int, num_slots: int) -> np.ndarray:
    """The `num_slots` most frequently routed bank ids l*E + e of a routing
    trace int [steps][L][k] (an id counted once per step and layer), most
    frequent first, ties to the lower id; ids never routed are not placed.

    A static cache hits an id once for every step and layer that routes it,
    so when the counts come from the trace that is then replayed no other
    fixed set of `num_slots` ids gets more hits on it: the static baseline is
    given hindsight."""
    tr = np.asarray(trace)
    if tr.ndim != 3:
        raise ValueError("trace must be [steps][L][k]")
    steps, L, k = tr.shape
    E = int(num_experts)
    if steps and (tr.min() < 0 or tr.max() >= E):
        raise ValueError("trace ids must lie in [0, num_experts)")
    counts = np.zeros(L * E, np.int64)
    for l in range(L):
        for t in range(steps):
            counts[l * E + np.unique(tr[t, l])] += 1
    order = np.lexsort((np.arange(L * E), -counts))  # count descending, then id ascending
    order = order[counts[order] > 0]
    return order[:max(int(num_slots), 0)].astype(np.int32)


def layer_placement(num_layers: int, num_experts: int, num_slots: int) -> np.ndarray:
    """Whole layers: every expert of layers 0 .. floor(S / E) - 1 (the slots
    left over hold nothing, as a layer is placed whole or not at all)."""
    n_layers = min(int(num_slots) // int(num_experts), int(num_layers))
    return np.arange(n_layers * int(num_experts), dtype=np.int32)
