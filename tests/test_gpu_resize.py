"""GPU parity of the elastic slot-pool re-division (moe_cache_resize; FreeToken
reader "Elastic Memory Management") against the oracle's cache_resize, through
the C ABI.

After every resize the tables (slot_of_id, id_of_slot, ts, clock) equal the
oracle's bit for bit, the evicted set and the (from, to) moves equal the
oracle's, and every resident slot holds its expert's bank blob byte for byte.
Decode steps between the resizes (moe_layer_forward, with the one-kernel step
where the shape allows it) keep matching the oracle's plans and outputs, so a
resize changes what is resident, never what is computed.
"""
import numpy as np
import pytest

import moe_expert_offload_gb300 as m
from moe_expert_offload_gb300 import synth

from gpu_util import assert_ffn_close, dev, dev_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_offload_gb300 import _build
    import oracle

    _build.build()
    oracle.build()
    m.lib()


@pytest.fixture(scope="module")
def oracle():
    import oracle as o

    return o


def _resize(cache, spec, S_new):
    wsb = m.moe_cache_resize_workspace_bytes(cache.c, S_new)
    ws = torch.full((wsb // 4,), -7, dtype=torch.int32, device=DEV)
    S_old = cache.c.num_slots
    m.moe_cache_resize(spec, cache.c, S_new, ws, wsb)
    assert cache.c.num_slots == S_new
    torch.cuda.synchronize()
    w = ws.cpu().numpy()
    cap = max(S_old, S_new)
    n_ev, n_mv = int(w[0]), int(w[1])
    return {"n_evicted": n_ev, "n_moved": n_mv, "n_occupied": int(w[2]), "err": int(w[3]),
            "move_from": w[8:8 + n_mv], "move_to": w[8 + cap:8 + cap + n_mv],
            "evicted_ids": w[8 + 2 * cap:8 + 2 * cap + n_ev]}


def _check_resize(got, want, cache, ost, bank_h):
    assert got["err"] == 0
    for key in ("n_evicted", "n_moved", "n_occupied"):
        assert got[key] == want[key], key
    # the device lists its evictions in slot order, the oracle in (ts, slot) order
    assert sorted(got["evicted_ids"]) == sorted(want["evicted_ids"])
    assert np.array_equal(got["move_from"], want["move_from"])
    assert np.array_equal(got["move_to"], want["move_to"])
    soi, ios, ts, clk = cache.host_tables()
    assert np.array_equal(soi, ost.slot_of_id)
    assert np.array_equal(ios, ost.id_of_slot)
    assert np.array_equal(ts, ost.ts)
    assert clk[0] == ost.clock[0]
    if bank_h is not None and cache.pool is not None:
        pool = cache.pool[:cache.c.num_slots].cpu().numpy()
        for slot, eid in enumerate(ost.id_of_slot):
            if eid >= 0:
                assert np.array_equal(pool[slot], bank_h[eid]), f"slot {slot}"


@pytest.mark.parametrize("seed", range(3))
def test_resize_tables_match_oracle_between_control_steps(oracle, seed):
    """Random traces through moe_cache_step (fills copied into the pool), with
    shrinks and growths between the steps, including one slot and growth past
    the starting size."""
    L, H, I, E, k, T, K = 3, 256, 128, 16, 2, 2, 4
    spec = m.make_spec(L, H, I, E, k)
    bank_h = synth.make_bank(L * E, H, I, 40 + seed)
    bank = dev(bank_h, DEV)
    cap, S = 40, 10
    cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=bank, device=DEV, capacity=cap)
    plan = m.DevicePlan(T * k, K, device=DEV)
    ost = oracle.CacheState(L * E, S)
    rng = np.random.default_rng(seed)
    sizes = [8, 12, 3, 1, 25, 40, 6, 6, 17]
    for j, S_new in enumerate(sizes):
        for _ in range(int(rng.integers(3, 9))):
            layer = int(rng.integers(0, L))
            ids_h = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(
                np.int32)
            m.moe_cache_step(spec, cache.c, layer, dev(ids_h, DEV), T, plan.c, 1)
            op = oracle.cache_step(ost, E, layer, ids_h, K, 52700, 77300)
            torch.cuda.synchronize()
            assert int(plan.counts[4].item()) == op["n_fill"]
        want = oracle.cache_resize(ost, S_new)
        got = _resize(cache, spec, S_new)
        _check_resize(got, want, cache, ost, bank_h)


def test_resize_worked_example_10_8_12(oracle):
    """The reader's sequence: 10 occupied slots, then 8 (two evicted), then 12
    (four new empty slots), with stamps set by steps that route every expert."""
    L, H, I, E, k, K = 1, 256, 128, 32, 1, 1
    spec = m.make_spec(L, H, I, E, k)
    bank_h = synth.make_bank(E, H, I, 5)
    bank = dev(bank_h, DEV)
    cache = m.DeviceCache(spec, 10, K, 100, 100, bank=bank, device=DEV, capacity=12)
    plan = m.DevicePlan(1, K, device=DEV)
    ost = oracle.CacheState(E, 10)
    # one expert per step: each fills the oldest slot (B_H = B_P: every miss filled)
    for e in (3, 9, 14, 1, 27, 8, 30, 2, 19, 11, 3, 27):
        ids_h = np.array([[e]], dtype=np.int32)
        m.moe_cache_step(spec, cache.c, 0, dev(ids_h, DEV), 1, plan.c, 1)
        oracle.cache_step(ost, E, 0, ids_h, K, 100, 100)
    torch.cuda.synchronize()
    assert np.all(ost.id_of_slot >= 0)
    want = oracle.cache_resize(ost, 8)
    got = _resize(cache, spec, 8)
    assert got["n_evicted"] == 2
    # the two least recently routed: 9 (step 2) and 14 (step 3)
    assert sorted(got["evicted_ids"]) == [9, 14]
    _check_resize(got, want, cache, ost, bank_h)
    want = oracle.cache_resize(ost, 12)
    got = _resize(cache, spec, 12)
    assert got["n_evicted"] == 0 and got["n_moved"] == 0 and got["n_occupied"] == 8
    _check_resize(got, want, cache, ost, bank_h)


def test_resize_rejects_a_broken_table_without_changes(oracle):
    """A slot table that is not a bijection (slot 0 claims an id whose entry
    points elsewhere) is reported in the workspace's error word and left as is."""
    L, H, I, E, k = 1, 256, 128, 16, 2
    spec = m.make_spec(L, H, I, E, k)
    cache = m.DeviceCache(spec, 6, 2, 52700, 77300, bank=None, device=DEV, with_pool=False)
    cache.id_of_slot[0] = 5  # slot_of_id[5] stays -1
    before = cache.host_tables()
    got = _resize(cache, spec, 3)
    assert got["err"] == m.MOE_DERR_RANGE and got["n_evicted"] == 0
    after = cache.host_tables()
    assert np.array_equal(before[0], after[0])
    assert np.array_equal(before[1][:3], after[1])


@pytest.mark.parametrize("sync", [True, False])
def test_layer_forward_across_resizes(oracle, sync):
    """moe_layer_forward between resizes: routing, plans and outputs equal the
    oracle's before and after each re-division (the one-kernel step with the
    cache's sync words), and resident slots hold their bank blobs."""
    L, H, I, E, k, T, K = 2, 1024, 512, 16, 4, 2, 3
    spec = m.make_spec(L, H, I, E, k, has_shared=True)
    bank_h = synth.make_bank(L * E + 1, H, I, 17)
    bank = dev(bank_h, DEV)
    cap, S = 16, 6
    cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=bank[:L * E], device=DEV, sync=sync,
                          capacity=cap)
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    ost = oracle.CacheState(L * E, S)
    rng = np.random.default_rng(3)
    step = 0
    for S_new in (4, 10, 2, 16, 7):
        for _ in range(4):
            layer = step % L
            wr_h = synth.router_weights(70 + layer, E, H)
            xb = synth.bf16_bits(rng.normal(0, 1.5, (T, H)))
            m.moe_layer_forward(spec, cache.c, layer, dev_bits(xb, DEV), T, dev_bits(wr_h, DEV),
                                None, bank[L * E], plan.c, ids, wts, ws, wsb, y)
            torch.cuda.synchronize()
            oid, ow = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h), k)
            assert np.array_equal(ids.cpu().numpy(), oid)
            op = oracle.cache_step(ost, E, layer, oid, K, 52700, 77300)
            gp = plan.read(K)
            for key in ("uniq", "hit_ids", "hit_slots", "fill_ids", "fill_slots", "evicted_ids",
                        "direct_ids", "victims", "counts"):
                assert np.array_equal(gp[key], op[key]), (step, key)
            ref = oracle.moe_ffn(list(bank_h[layer * E:(layer + 1) * E]), H, I, xb, oid, ow,
                                 bank_h[L * E], I)
            assert_ffn_close(y.cpu().numpy(), ref, f"step {step}")
            step += 1
        want = oracle.cache_resize(ost, S_new)
        got = _resize(cache, spec, S_new)
        _check_resize(got, want, cache, ost, bank_h)
    assert int(plan.err[0].item()) == 0
    if sync:
        assert not cache.sync.any().item()
