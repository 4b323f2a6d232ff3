"""Pins of the oracle's elastic slot-pool re-division (FreeToken reader,
"Elastic Memory Management") against the page's worked example and against
an independent brute-force restatement of the reading: on a shrink the
occupied slots with the smallest (ts, slot) keys are evicted until S_new
remain, the kept experts past S_new move to the free slots below it in
ascending order with their ts, and the slots past the smaller size are empty.
"""
import os

import numpy as np
import pytest

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    for line in open(os.path.join(GOLD, name)):
        line = line.split("#")[0].strip()
        if line:
            out.append(line.split())
    return out


@pytest.fixture(scope="module")
def oracle():
    import oracle as o

    o.build()
    return o


def _random_state(oracle, rng, n_ids, S, fill, ts_max=50):
    st = oracle.CacheState(n_ids, S)
    slots = rng.permutation(S)[:int(round(fill * S))]
    ids = rng.choice(n_ids, size=slots.size, replace=False)
    for v, u in zip(slots, ids):
        st.id_of_slot[v] = u
        st.slot_of_id[u] = v
        st.ts[v] = rng.integers(1, ts_max)
    st.clock[0] = ts_max
    return st


def _brute(slot_of_id, id_of_slot, ts, S_new):
    """The reading restated with Python lists: kept = the S_new occupied
    entries with the largest (ts, slot) keys; returns {id: ts} kept and the
    evicted ids in (ts, slot) order."""
    occ = sorted((int(ts[v]), v, int(id_of_slot[v])) for v in range(id_of_slot.size)
                 if id_of_slot[v] >= 0)
    n_ev = max(0, len(occ) - S_new)
    return {u: t for t, _, u in occ[n_ev:]}, [u for _, _, u in occ[:n_ev]]


def _check_tables(st, n_ids):
    S = st.id_of_slot.size
    for v in range(S):
        u = st.id_of_slot[v]
        if u >= 0:
            assert st.slot_of_id[u] == v
        else:
            assert st.ts[v] == 0
    for u in range(n_ids):
        v = st.slot_of_id[u]
        if v >= 0:
            assert v < S and st.id_of_slot[v] == u


def test_slots_for_budget_worked_example(oracle):
    for free_gb, slot_gb, want in _rows("elastic_slots.txt"):
        free = int(float(free_gb) * 2**30)
        slot = int(float(slot_gb) * 2**30)
        assert oracle.slots_for_budget(free, slot) == int(want)
    assert oracle.slots_for_budget(0, 7) == 0
    assert oracle.slots_for_budget(13, 7) == 1
    with pytest.raises(ValueError):
        oracle.slots_for_budget(10, 0)


def test_worked_example_10_8_12(oracle):
    """10 slots all holding experts, then 8 (two evicted: the two least
    recently routed), then 12 (four new empty slots; nothing evicted)."""
    rows = _rows("elastic_slots.txt")
    sizes = [int(r[2]) for r in rows]
    n_ids = 64
    st = oracle.CacheState(n_ids, sizes[0])
    ids = np.arange(sizes[0]) * 5 + 1
    oracle.cache_place(st, n_ids, 1, ids)
    stamps = np.array([9, 3, 14, 8, 11, 2, 13, 10, 12, 7], dtype=np.uint32)
    st.ts[:] = stamps
    r = oracle.cache_resize(st, sizes[1])
    assert r["n_evicted"] == sizes[0] - sizes[1] == 2
    # the two smallest stamps: slot 5 (ts 2) then slot 1 (ts 3)
    assert list(r["evicted_ids"]) == [int(ids[5]), int(ids[1])]
    assert st.id_of_slot.size == 8 and r["n_occupied"] == 8
    kept = {int(ids[v]): int(stamps[v]) for v in range(10) if v not in (1, 5)}
    assert {int(st.id_of_slot[v]): int(st.ts[v]) for v in range(8)} == kept
    # slots 8 and 9 moved into the freed slots 1 and 5, in that order
    assert list(r["move_from"]) == [8, 9] and list(r["move_to"]) == [1, 5]
    _check_tables(st, n_ids)
    before = st.id_of_slot.copy(), st.ts.copy(), st.slot_of_id.copy()
    r = oracle.cache_resize(st, sizes[2])
    assert r["n_evicted"] == 0 and r["n_moved"] == 0 and r["n_occupied"] == 8
    assert np.array_equal(st.id_of_slot[:8], before[0]) and np.array_equal(st.ts[:8], before[1])
    assert np.all(st.id_of_slot[8:] == -1) and np.all(st.ts[8:] == 0)
    assert np.array_equal(st.slot_of_id, before[2])


@pytest.mark.parametrize("seed", range(12))
def test_resize_matches_brute_force(oracle, seed):
    rng = np.random.default_rng(seed)
    n_ids = 200
    S = int(rng.integers(1, 60))
    st = _random_state(oracle, rng, n_ids, S, fill=float(rng.uniform(0, 1)),
                       ts_max=int(rng.choice([3, 50])))  # few stamps: many ties
    for _ in range(4):
        S_new = int(rng.integers(1, 80))
        want_kept, want_ev = _brute(st.slot_of_id, st.id_of_slot, st.ts, S_new)
        old_slot = st.slot_of_id.copy()
        r = oracle.cache_resize(st, S_new)
        assert list(r["evicted_ids"]) == want_ev
        got = {int(st.id_of_slot[v]): int(st.ts[v]) for v in range(S_new) if st.id_of_slot[v] >= 0}
        assert got == want_kept
        # only the experts past S_new moved, into free slots below it, in order
        assert all(f >= S_new for f in r["move_from"]) and all(t < S_new for t in r["move_to"])
        assert list(r["move_from"]) == sorted(r["move_from"])
        assert list(r["move_to"]) == sorted(r["move_to"])
        for u in want_kept:
            if old_slot[u] < S_new:
                assert st.slot_of_id[u] == old_slot[u]
        _check_tables(st, n_ids)
        S = S_new


def test_resize_then_step_takes_new_slots_first(oracle):
    """After a growth the new slots are empty (ts 0), so the next step's
    victim scan hands them out before any occupied slot."""
    E, S, K = 32, 4, 4
    st = oracle.CacheState(E, S)
    oracle.cache_place(st, E, 1, [0, 1, 2, 3])
    st.ts[:] = [1, 2, 3, 4]
    st.clock[0] = 4
    oracle.cache_resize(st, 7)
    plan = oracle.cache_step(st, E, 0, np.array([10, 11]), K, 100, 100)
    assert list(plan["victims"]) == [4, 5, 6, 0]
    assert list(plan["fill_slots"]) == [4, 5]


def test_resize_rejects_bad_sizes_and_tables(oracle):
    st = oracle.CacheState(8, 4)
    with pytest.raises(ValueError):
        oracle.cache_resize(st, 0)
    st.id_of_slot[0] = 3  # slot 0 claims id 3, but id 3 has no slot
    with pytest.raises(ValueError):
        oracle.cache_resize(st.copy(), 2)
