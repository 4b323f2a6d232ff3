"""Property checks of the oracle's control step under every replacement policy
(FreeToken summary "method steps"; Edge0 §3.1 "hot" path), on random shapes
and traces.  Each property is derived from the step's definition, not from the
oracle's code: a partition of the routed set, F as a prefix of the ascending
misses, victims as the K smallest (ts, slot) keys of the policy's slot range
taken from the tables before the step, and the tables staying a bijection."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")

POLICIES = (0, 1, 2)  # shared LRU, per-layer LRU, static placement


@hyp.settings(max_examples=60, deadline=None)
@hyp.given(seed=st.integers(0, 2**31 - 1), policy=st.sampled_from(POLICIES),
           L=st.integers(1, 4), E=st.integers(2, 12), K=st.integers(1, 8),
           bpbh=st.sampled_from([(52700, 77300), (11800, 47500), (77300, 77300), (9, 4)]))
def test_control_step_properties(oracle, seed, policy, L, E, K, bpbh):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(L, 3 * L * E + 1))
    bp, bh = bpbh
    stt = oracle.CacheState(L * E, S)
    if policy == 2 or rng.random() < 0.5:
        Sl = S // L if policy == 1 else S
        per = [l * E + int(e) for l in range(L)
               for e in rng.choice(E, size=min(E, Sl if policy == 1 else max(1, S // L)),
                                   replace=False)]
        if policy != 1:
            per = per[:S]
        oracle.cache_place(stt, E, L, per, policy=policy)
    placed = set(int(u) for u in np.nonzero(stt.slot_of_id >= 0)[0])
    for step in range(25):
        layer = int(rng.integers(L))
        T = int(rng.integers(1, 4))
        ids = rng.integers(0, E, size=(T, min(E, 3)))
        before_ts = stt.ts.copy()
        before_soi = stt.slot_of_id.copy()
        plan = oracle.cache_step(stt, E, layer, ids, K, bp, bh, policy=policy, L=L)
        now = plan["now"]
        U = sorted({layer * E + int(i) for i in ids.reshape(-1)})
        assert list(plan["uniq"]) == U
        Hs = [u for u in U if before_soi[u] >= 0]
        M = [u for u in U if before_soi[u] < 0]
        assert list(plan["hit_ids"]) == Hs
        assert list(plan["hit_slots"]) == [int(before_soi[u]) for u in Hs]
        F, C = list(plan["fill_ids"]), list(plan["direct_ids"])
        assert F + C == M  # F is a prefix of the ascending misses
        # victims: the K smallest (ts, slot) over the range, hits excluded
        lo, hi = (layer * (S // L), layer * (S // L) + S // L) if policy == 1 else (0, S)
        hit_slots = {int(before_soi[u]) for u in Hs}
        keys = sorted((int(before_ts[v]), v) for v in range(lo, hi) if v not in hit_slots)
        assert [v for v in plan["victims"] if v >= 0] == [v for _, v in keys[:K]]
        assert list(plan["fill_slots"]) == [v for _, v in keys[:len(F)]]
        if policy == 2:
            assert F == [] and plan["q"] == 0
            assert set(int(u) for u in np.nonzero(stt.slot_of_id >= 0)[0]) == placed
        # the tables stay a bijection between resident ids and used slots
        used = np.nonzero(stt.id_of_slot >= 0)[0]
        assert np.all(stt.slot_of_id[stt.id_of_slot[used]] == used)
        assert int(np.sum(stt.slot_of_id >= 0)) == len(used)
        for u in Hs + F:
            assert stt.ts[stt.slot_of_id[u]] == now
        if policy == 1:
            for v in used:
                assert v < L * (S // L) and stt.id_of_slot[v] // E == v // (S // L)
