"""GPU parity of the decode path against the CPU oracle, through the C ABI.

Routing (logits, ids, weights), the control step (sets, victims, tables) and
the slot-pool contents must match bit for bit; expert-FFN outputs must be
within the Edge0 tolerance (relative L2 <= 1e-2, |err| <= 2e-2 * max|y|).
"""
import time

import numpy as np
import pytest

import moe_expert_offload_gb300 as m
from moe_expert_offload_gb300 import synth

from gpu_util import assert_ffn_close, dev, dev_bits, f32_bits

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


# ------------------------------------------------------------------ routing
def _route(spec, xb, wb, bias=None):
    T = xb.shape[0]
    E, k = spec.num_experts, spec.top_k
    x = dev_bits(xb, DEV)
    w = dev_bits(wb, DEV)
    b = None if bias is None else dev(bias, DEV)
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    m.moe_route(spec, x, T, w, b, logits, ids, wts)
    torch.cuda.synchronize()
    return logits.cpu().numpy(), ids.cpu().numpy(), wts.cpu().numpy()


@pytest.mark.parametrize("T,E,H,k", [(1, 16, 256, 2), (1, 256, 2048, 8), (8, 256, 2048, 8),
                                     (8, 256, 7168, 8), (5, 20, 320, 3), (3, 1000, 64, 7),
                                     (64, 64, 512, 4), (37, 40, 512, 5), (512, 256, 2048, 8)])
def test_softmax_routing_bit_exact(oracle, T, E, H, k):
    rng = np.random.default_rng(T * 1000 + E)
    xb = synth.bf16_bits(rng.normal(0, 2.3, (T, H)))
    wb = synth.router_weights(E + H, E, H)
    spec = m.make_spec(1, max(H, 64) // 64 * 64, 64, E, k)
    spec.hidden = H
    lg, ids, w = _route(spec, xb, wb)
    ol = oracle.router_logits(xb, wb)
    assert np.array_equal(f32_bits(lg), f32_bits(ol))
    oid, ow = oracle.route_softmax_topk(ol, k)
    assert np.array_equal(ids, oid)
    assert np.array_equal(f32_bits(w), f32_bits(ow))


def test_softmax_routing_ties(oracle):
    # experts 3, 7 and 11 share one router row: equal logits, lower index ranks first
    T, E, H, k = 4, 16, 256, 4
    rng = np.random.default_rng(5)
    wb = synth.router_weights(9, E, H)
    wb[7] = wb[3]
    wb[11] = wb[3]
    xb = synth.bf16_bits(rng.normal(0, 1, (T, H)))
    xb[0] = synth.bf16_bits(synth.bf16_value(wb[3]) * 50)  # token 0 prefers the tied rows
    spec = m.make_spec(1, H, 64, E, k)
    lg, ids, w = _route(spec, xb, wb)
    ol = oracle.router_logits(xb, wb)
    oid, ow = oracle.route_softmax_topk(ol, k)
    assert list(ids[0][:3]) == [3, 7, 11]
    assert np.array_equal(ids, oid) and np.array_equal(f32_bits(w), f32_bits(ow))


@pytest.mark.parametrize("T,E,H,ng,G,k,scale", [(1, 256, 7168, 8, 4, 8, 2.5),
                                                 (40, 256, 7168, 8, 4, 8, 2.5),
                                                 (8, 256, 7168, 8, 4, 8, 2.5),
                                                 (16, 16, 256, 4, 2, 3, 1.0),
                                                 (7, 64, 512, 32, 3, 4, 2.0)])
def test_sigmoid_group_routing_bit_exact(oracle, T, E, H, ng, G, k, scale):
    rng = np.random.default_rng(E + T)
    xb = synth.bf16_bits(rng.normal(0, 2.3, (T, H)))
    wb = synth.router_weights(E * 7 + H, E, H)
    bias = synth.selection_bias(3, E)
    spec = m.make_spec(1, H, 64, E, k, router="sigmoid_group", n_groups=ng, topk_groups=G,
                       routed_scale=scale)
    lg, ids, w = _route(spec, xb, wb, bias)
    ol = oracle.router_logits(xb, wb)
    assert np.array_equal(f32_bits(lg), f32_bits(ol))
    oid, ow = oracle.route_sigmoid_group(ol, bias, ng, G, k, scale)
    assert np.array_equal(ids, oid)
    assert np.array_equal(f32_bits(w), f32_bits(ow))


def test_exp_sweep_through_softmax_weights(oracle):
    # two experts per token with logit gap d: weight[1] = e^-d / (1 + e^-d) uses the
    # library's own exp; a dense sweep of gaps compares it bit for bit.
    T, E, H = 4096, 2, 64
    gaps = np.linspace(0, 60, T).astype(np.float32)
    wb = np.zeros((E, H), np.uint16)
    wb[0, 0] = synth.bf16_bits([1.0])[0]
    xb = synth.bf16_bits(gaps[:, None] * (np.arange(H) == 0))
    spec = m.make_spec(1, H, 64, E, 2)
    lg, ids, w = _route(spec, xb, wb)
    ol = oracle.router_logits(xb, wb)
    oid, ow = oracle.route_softmax_topk(ol, 2)
    assert np.array_equal(ids, oid) and np.array_equal(f32_bits(w), f32_bits(ow))


# ---------------------------------------------------------- control step
def _tables_equal(cache, ost):
    soi, ios, ts, clk = cache.host_tables()
    assert np.array_equal(soi, ost.slot_of_id)
    assert np.array_equal(ios, ost.id_of_slot)
    assert np.array_equal(ts, ost.ts)
    assert clk[0] == ost.clock[0]


def _plans_equal(gp, op, K):
    for key in ("uniq", "hit_ids", "hit_slots", "fill_ids", "fill_slots", "evicted_ids",
                "direct_ids", "victims"):
        assert np.array_equal(gp[key], op[key]), key
    assert np.array_equal(gp["counts"], op["counts"])


@pytest.mark.parametrize("L,E,S,K,bp,bh,T,k,steps", [
    (1, 16, 8, 4, 52700, 77300, 1, 2, 64),       # tiny decode config
    (3, 16, 5, 3, 11800, 47500, 4, 2, 120),
    (2, 32, 1, 1, 77300, 77300, 1, 4, 60),       # one slot, pure fill
    (2, 32, 40, 8, 60000, 50000, 8, 8, 80),      # B_H < B_P -> pure fill
    (4, 64, 7, 16, 1, 1000, 8, 8, 80),           # K > S, q mostly 0
    (2, 64, 40, 20, 52700, 77300, 2, 8, 60),     # K > 16: the long victim lists
])
def test_cache_step_matches_oracle_on_random_traces(oracle, L, E, S, K, bp, bh, T, k, steps):
    rng = np.random.default_rng(S * 31 + K)
    spec = m.make_spec(L, 64, 64, E, k)
    cache = m.DeviceCache(spec, S, K, bp, bh, bank=None, device=DEV, with_pool=False)
    plan = m.DevicePlan(T * k, K, device=DEV)
    ost = oracle.CacheState(L * E, S)
    for step in range(steps):
        layer = step % L
        ids_h = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        ids = dev(ids_h, DEV)
        m.moe_cache_step(spec, cache.c, layer, ids, T, plan.c, do_fill=0)
        torch.cuda.synchronize()
        op = oracle.cache_step(ost, E, layer, ids_h, K, bp, bh)
        _plans_equal(plan.read(K), op, K)
        _tables_equal(cache, ost)


@pytest.mark.parametrize("S,bp,bh", [(512, 52700, 77300), (5120, 52700, 77300),
                                     (2560, 11800, 47500), (2560, 77300, 77300)])
def test_cache_step_zipf_trace_sweep_shape(oracle, S, bp, bh):
    """The cache sweep's shape (40 layers x 256 experts, top-8 Zipf traces with step
    overlap, K=8) over 64 steps at each B_P/B_H pair of the sweep: plans every 13th layer
    and all tables after every step, bit for bit."""
    L, E, k, K, steps = 40, 256, 8, 8, 64
    spec = m.make_spec(L, 64, 64, E, k)
    cache = m.DeviceCache(spec, S, K, bp, bh, bank=None, device=DEV, with_pool=False)
    plan = m.DevicePlan(k, K, device=DEV)
    ost = oracle.CacheState(L * E, S)
    traces = [synth.zipf_trace(1000 + l, steps, E, k) for l in range(L)]
    fills = 0
    for s in range(steps):
        for layer in range(L):
            ids_h = traces[layer][s:s + 1]
            m.moe_cache_step(spec, cache.c, layer, dev(ids_h, DEV), 1, plan.c, do_fill=0)
            op = oracle.cache_step(ost, E, layer, ids_h, K, bp, bh)
            fills += op["n_fill"]
            if layer % 13 == 0:
                torch.cuda.synchronize()
                _plans_equal(plan.read(K), op, K)
        torch.cuda.synchronize()
        _tables_equal(cache, ost)
    assert fills > 0


def test_cache_step_all_hits_then_duplicates(oracle):
    L, E, S, K, k = 1, 16, 16, 4, 4
    spec = m.make_spec(L, 64, 64, E, k)
    cache = m.DeviceCache(spec, S, K, 77300, 77300, bank=None, device=DEV, with_pool=False)
    plan = m.DevicePlan(2 * k, K, device=DEV)
    ost = oracle.CacheState(E, S)
    seq = [np.array([[0, 1, 2, 3]]), np.array([[0, 1, 2, 3]]),
           np.array([[3, 2, 1, 0], [0, 5, 1, 6]])]
    for ids_h in seq:
        ids_h = ids_h.astype(np.int32)
        T = ids_h.shape[0]
        m.moe_cache_step(spec, cache.c, 0, dev(ids_h, DEV), T, plan.c, do_fill=0)
        torch.cuda.synchronize()
        op = oracle.cache_step(ost, E, 0, ids_h, K, 77300, 77300)
        gp = plan.read(K)
        _plans_equal(gp, op, K)
    assert gp["n_uniq"] == 6 and gp["n_hit"] == 4 and gp["n_fill"] == 2


def test_cache_step_flags_bad_ids(oracle):
    E, S, K, k = 16, 8, 4, 2
    spec = m.make_spec(1, 64, 64, E, k)
    cache = m.DeviceCache(spec, S, K, 77300, 77300, bank=None, device=DEV, with_pool=False)
    plan = m.DevicePlan(4, K, device=DEV)
    ids_h = np.array([[3, 99], [-2, 5]], np.int32)
    m.moe_cache_step(spec, cache.c, 0, dev(ids_h, DEV), 2, plan.c, do_fill=0)
    torch.cuda.synchronize()
    gp = plan.read(K)
    assert gp["err"] & m.MOE_DERR_BAD_ID
    ost = oracle.CacheState(E, S)
    op = oracle.cache_step(ost, E, 0, np.array([3, 5], np.int32), K, 77300, 77300)
    _plans_equal(gp, op, K)


# ------------------------------------------------------- replacement policies
def _placement(rng, policy, L, E, S):
    """A random warm-start / static set in shuffled order (at most S_l per layer)."""
    if policy == m.POLICY_LAYER_LRU:
        Sl = S // L
        ids = [l * E + int(e) for l in range(L)
               for e in rng.choice(E, size=int(rng.integers(0, min(Sl, E) + 1)), replace=False)]
    else:
        ids = [int(u) for u in rng.choice(L * E, size=min(S, L * E) - 1, replace=False)]
    rng.shuffle(ids)
    return np.array(ids, np.int32)


@pytest.mark.parametrize("policy,L,E,S,K,T,k,steps", [
    (m.POLICY_LAYER_LRU, 3, 16, 14, 3, 2, 2, 40),       # S_l = 4; slots 12, 13 unused
    (m.POLICY_LAYER_LRU, 40, 256, 5120, 8, 1, 8, 3),    # ranges past the early-loaded slots
    (m.POLICY_LAYER_LRU, 2, 64, 90, 20, 2, 8, 30),      # K > 16: the long victim lists
    (m.POLICY_LAYER_LRU, 4, 16, 4, 1, 1, 2, 20),        # one slot per layer
    (m.POLICY_STATIC, 3, 16, 20, 4, 2, 3, 30),
    (m.POLICY_STATIC, 40, 256, 2560, 8, 1, 8, 3),
])
def test_cache_policies_match_oracle(oracle, policy, L, E, S, K, T, k, steps):
    """Per-layer LRU and static placement: plans and tables equal the oracle's after a
    placement and over random multi-layer traces (layers in random order)."""
    rng = np.random.default_rng(S + 7 * K + policy)
    spec = m.make_spec(L, 64, 64, E, k)
    cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=None, device=DEV, with_pool=False,
                          policy=policy)
    plan = m.DevicePlan(T * k, K, device=DEV)
    ost = oracle.CacheState(L * E, S)
    placed = _placement(rng, policy, L, E, S)
    m.moe_cache_place(spec, cache.c, placed)
    oracle.cache_place(ost, E, L, placed, policy=policy)
    _tables_equal(cache, ost)
    for it in range(steps * L):
        layer = int(rng.integers(L))
        ids_h = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        m.moe_cache_step(spec, cache.c, layer, dev(ids_h, DEV), T, plan.c, do_fill=0)
        torch.cuda.synchronize()
        op = oracle.cache_step(ost, E, layer, ids_h, K, 52700, 77300, policy=policy, L=L)
        _plans_equal(plan.read(K), op, K)
        if it % 16 == 0:
            _tables_equal(cache, ost)
    _tables_equal(cache, ost)


@pytest.mark.parametrize("policy", [m.POLICY_LAYER_LRU, m.POLICY_STATIC])
def test_layer_forward_under_policies(oracle, policy):
    """Whole decode layer step under each policy: routing, plans and FFN output equal the
    oracle's, and every resident slot holds its expert's bank blob (placement copies and
    per-layer fills)."""
    L, H, I, E, k, S, K, T = 2, 256, 128, 16, 2, 7, 2, 2   # per-layer: S_l = 3, slot 6 unused
    spec, bank, bank_h, cache, _ = _layer_rig(L, H, I, E, k, S, K, 52700, 77300, False, seed=9)
    cache.c.policy = policy
    rng = np.random.default_rng(policy)
    placed = _placement(rng, policy, L, E, S)
    m.moe_cache_place(spec, cache.c, placed)
    ost = oracle.CacheState(L * E, S)
    oracle.cache_place(ost, E, L, placed, policy=policy)
    pool = cache.pool.cpu().numpy()
    for slot, eid in enumerate(ost.id_of_slot):
        if eid >= 0:
            assert np.array_equal(pool[slot], bank_h[eid])
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    hits = 0
    for step in range(12):
        layer = step % L
        wr_h = synth.router_weights(30 + layer, E, H)
        xb = synth.bf16_bits(rng.normal(0, 1.5, (T, H)))
        m.moe_layer_forward(spec, cache.c, layer, dev_bits(xb, DEV), T, dev_bits(wr_h, DEV), None,
                            None, plan.c, ids, wts, ws, wsb, y)
        torch.cuda.synchronize()
        oid, ow = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h), k)
        assert np.array_equal(ids.cpu().numpy(), oid)
        op = oracle.cache_step(ost, E, layer, oid, K, 52700, 77300, policy=policy, L=L)
        _plans_equal(plan.read(K), op, K)
        hits += op["n_hit"]
        ref = oracle.moe_ffn(list(bank_h[layer * E:(layer + 1) * E]), H, I, xb, oid, ow)
        assert_ffn_close(y.cpu().numpy(), ref, f"policy {policy} step {step}")
    _tables_equal(cache, ost)
    pool = cache.pool.cpu().numpy()
    for slot, eid in enumerate(ost.id_of_slot):
        if eid >= 0:
            assert np.array_equal(pool[slot], bank_h[eid])
    assert hits > 0


# --------------------------------------------- fill carried by the decode FFN
def _ffn_kernels(H, I, T):
    """FFN launches of a decode layer step: one cooperative kernel where it serves the shape
    (H % 1024 == 0, I % 512 == 0, T <= 8), else the streaming gate/up and down kernels."""
    return 1 if (H % 1024 == 0 and I % 512 == 0 and T <= 8) else 2


def _layer_kernels(H, I, E, k, T, K, sync):
    """Launches of a decode layer step whose selection runs in the control step and whose
    fill the FFN carries: the whole step as one cooperative kernel when the cache has sync
    words and T k <= 32, K <= 8, E <= 256 on a cooperative-FFN shape; else logits, control
    step and the FFN kernels."""
    if sync and _ffn_kernels(H, I, T) == 1 and T * k <= 32 and K <= 8 and E <= 256:
        return 1
    return 2 + _ffn_kernels(H, I, T)


@pytest.mark.parametrize("H,I,E,k,T,shared,S,K", [(1024, 256, 16, 4, 1, True, 6, 3),
                                                  (1024, 256, 16, 4, 3, False, 5, 4),
                                                  (2048, 512, 24, 8, 8, True, 20, 8),
                                                  (512, 256, 12, 3, 2, True, 4, 2),
                                                  (1024, 512, 16, 4, 1, True, 6, 3),
                                                  (1024, 512, 16, 4, 3, False, 5, 4),
                                                  (2048, 1024, 12, 4, 8, True, 10, 4),
                                                  (3072, 512, 20, 6, 5, True, 8, 6)])
@pytest.mark.parametrize("sync", [True, False])
def test_layer_forward_fused_fill(oracle, H, I, E, k, T, shared, S, K, sync):
    """Shapes the FFN kernels serve with the fill carried: the fill copy is written by the
    FFN kernels as they read F from the bank (no copy kernel).  Plans, outputs and every
    resident slot's bytes equal the oracle's and the bank's over steps with fills and
    evictions.  The shapes cover both FFN paths (cooperative kernel: H % 1024 == 0 and
    I % 512 == 0), both down-tile geometries of the cooperative kernel (I % 1024 == 0 or
    not) and gate/up tiles of one, two and three stages.  With the cache's sync words
    (sync) the shapes with T k <= 32 run as one cooperative kernel (router logits,
    selection, control step and FFN); without them as logits, control step and FFN."""
    L = 2
    spec, bank, bank_h, cache, sh = _layer_rig(L, H, I, E, k, S, K, 52700, 77300, shared,
                                               seed=H + T, sync=sync)
    assert m.moe_layer_kernel_count(spec, cache.c, T) == _layer_kernels(H, I, E, k, T, K, sync)
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    ost = oracle.CacheState(L * E, S)
    rng = np.random.default_rng(T * 7 + S)
    fills = 0
    for step in range(10):
        layer = step % L
        wr_h = synth.router_weights(50 + layer, E, H)
        xb = synth.bf16_bits(rng.normal(0, 1.5, (T, H)))
        m.moe_layer_forward(spec, cache.c, layer, dev_bits(xb, DEV), T, dev_bits(wr_h, DEV), None,
                            sh, plan.c, ids, wts, ws, wsb, y)
        torch.cuda.synchronize()
        oid, ow = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h), k)
        assert np.array_equal(ids.cpu().numpy(), oid)
        op = oracle.cache_step(ost, E, layer, oid, K, 52700, 77300)
        _plans_equal(plan.read(K), op, K)
        fills += op["n_fill"]
        ref = oracle.moe_ffn(list(bank_h[layer * E:(layer + 1) * E]), H, I, xb, oid, ow,
                             bank_h[L * E] if shared else None, I)
        assert_ffn_close(y.cpu().numpy(), ref, f"step {step}")
        pool = cache.pool.cpu().numpy()
        for slot, eid in enumerate(ost.id_of_slot):
            if eid >= 0:
                assert np.array_equal(pool[slot], bank_h[eid]), f"step {step} slot {slot}"
    assert fills > 0
    assert int(plan.err[0].item()) == 0
    if sync:
        assert not cache.sync.any().item()  # every step leaves the sync words zero


# ------------------------------------------------ failure detection (no fault)
def test_ffn_wait_timeout_sets_error_and_context_survives(oracle):
    """The injected stall leaves the gate/up stages unfilled: the kernel's bounded waits
    (one second of device time) run out, plan.err gets MOE_DERR_WAIT and the call returns;
    the next call on the same context is correct."""
    H, I, E, k, T, S, K = 1024, 256, 16, 4, 1, 6, 3
    spec, bank, bank_h, cache, sh = _layer_rig(1, H, I, E, k, S, K, 52700, 77300, True, seed=5)
    plan = m.DevicePlan(T * k, K, device=DEV)
    fws = m.moe_ffn_workspace_bytes(spec, T)
    ws = torch.empty(fws, dtype=torch.uint8, device=DEV)
    ids_h = np.array([[1, 5, 9, 12]], np.int32)
    wts_h = np.array([[0.4, 0.3, 0.2, 0.1]], np.float32)
    ids, wts = dev(ids_h, DEV), dev(wts_h, DEV)
    xb = synth.bf16_bits(np.random.default_rng(0).normal(0, 1, (T, H)))
    x = dev_bits(xb, DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    m.moe_cache_step(spec, cache.c, 0, ids, T, plan.c, do_fill=1)
    torch.cuda.synchronize()
    m.moe_debug_inject_ffn_stall(True)
    t0 = time.perf_counter()
    m.moe_expert_ffn(spec, cache.c, 0, plan.c, x, T, ids, wts, sh, ws, fws, y)
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert plan.read(K)["err"] & m.MOE_DERR_WAIT
    assert 0.5 < took < 30.0, took
    plan.err.zero_()
    m.moe_expert_ffn(spec, cache.c, 0, plan.c, x, T, ids, wts, sh, ws, fws, y)
    torch.cuda.synchronize()
    assert int(plan.err[0].item()) == 0
    ref = oracle.moe_ffn(list(bank_h[:E]), H, I, xb, ids_h, wts_h, bank_h[E], I)
    assert_ffn_close(y.cpu().numpy(), ref, "after the stall")


@pytest.mark.parametrize("sync", [True, False])
def test_wait_timeout_in_layer_step_unmaps_fills(oracle, sync):
    """A decode layer step whose FFN carries the fill and whose bounded waits run out
    (injected stall): plan.err gets MOE_DERR_WAIT, and the experts the step filled are
    unmapped again (their slots may hold a partial copy): slot_of_id = -1, the slot empty,
    ts 0.  With the same edit applied to the oracle's tables, the following steps match the
    oracle bit for bit (plans, tables) and within tolerance (outputs), and every resident
    slot holds its bank blob."""
    H, I, E, k, T, S, K, L = 1024, 512, 16, 4, 1, 6, 3, 1
    spec, bank, bank_h, cache, sh = _layer_rig(L, H, I, E, k, S, K, 52700, 77300, True, seed=9,
                                               sync=sync)
    # one kernel for the whole step, or logits, control step and the cooperative FFN
    assert m.moe_layer_kernel_count(spec, cache.c, T) == (1 if sync else 3)
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    wr_h = synth.router_weights(21, E, H)
    wr = dev_bits(wr_h, DEV)
    ost = oracle.CacheState(L * E, S)
    rng = np.random.default_rng(4)
    stalled_fills = 0
    for step in range(8):
        xb = synth.bf16_bits(rng.normal(0, 1.5, (T, H)))
        stall = step == 3
        if stall:
            m.moe_debug_inject_ffn_stall(True)
        t0 = time.perf_counter()
        m.moe_layer_forward(spec, cache.c, 0, dev_bits(xb, DEV), T, wr, None, sh, plan.c, ids,
                            wts, ws, wsb, y)
        torch.cuda.synchronize()
        took = time.perf_counter() - t0
        oid, ow = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h), k)
        assert np.array_equal(ids.cpu().numpy(), oid)
        op = oracle.cache_step(ost, E, 0, oid, K, 52700, 77300)
        gp = plan.read(K)
        _plans_equal(gp, op, K)
        if stall:
            assert gp["err"] & m.MOE_DERR_WAIT
            assert 0.5 < took < 30.0, took
            stalled_fills = op["n_fill"]
            for f, v in zip(op["fill_ids"][:op["n_fill"]], op["fill_slots"][:op["n_fill"]]):
                ost.slot_of_id[f] = -1
                ost.id_of_slot[v] = -1
                ost.ts[v] = 0
            plan.err.zero_()
        else:
            assert gp["err"] == 0
            ref = oracle.moe_ffn(list(bank_h[:E]), H, I, xb, oid, ow, bank_h[E], I)
            assert_ffn_close(y.cpu().numpy(), ref, f"step {step}")
        _tables_equal(cache, ost)
        pool = cache.pool.cpu().numpy()
        for slot, eid in enumerate(ost.id_of_slot):
            if eid >= 0:
                assert np.array_equal(pool[slot], bank_h[eid]), f"step {step} slot {slot}"
    assert stalled_fills > 0, "the stalled step filled nothing: pick another seed"


# ------------------------------------------------------- fill + expert FFN
def _layer_rig(L, H, I, E, k, S, K, bp, bh, has_shared, seed=0, big=False, sync=True):
    spec = m.make_spec(L, H, I, E, k, has_shared=has_shared)
    if big:
        bank = synth.make_bank_torch(L * E + 1, H, I, seed, DEV)
        bank_h = None
    else:
        bank_h = synth.make_bank(L * E + 1, H, I, seed)
        bank = dev(bank_h, DEV)
    cache = m.DeviceCache(spec, S, K, bp, bh, bank=bank[:L * E], device=DEV, sync=sync)
    shared = bank[L * E] if has_shared else None
    return spec, bank, bank_h, cache, shared


def test_tiny_config_64_decode_steps(oracle):
    """Tiny single layer (H=256, I=128, E=16, top-2), AR(1) inputs, 64 steps, S=8, K=4."""
    H, I, E, k, S, K, T = 256, 128, 16, 2, 8, 4, 1
    spec, bank, bank_h, cache, _ = _layer_rig(1, H, I, E, k, S, K, 52700, 77300, False)
    wr_h = synth.router_weights(0, E, H)
    wr = dev_bits(wr_h, DEV)
    xs = synth.ar1_stream(0, 64, H)
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    ost = oracle.CacheState(E, S)
    fills = 0
    for step in range(64):
        xb = xs[step]
        m.moe_layer_forward(spec, cache.c, 0, dev_bits(xb, DEV), T, wr, None, None, plan.c, ids,
                            wts, ws, wsb, y)
        torch.cuda.synchronize()
        oid, ow = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h), k)
        assert np.array_equal(ids.cpu().numpy(), oid)
        assert np.array_equal(f32_bits(wts.cpu().numpy()), f32_bits(ow))
        op = oracle.cache_step(ost, E, 0, oid, K, 52700, 77300)
        _plans_equal(plan.read(K), op, K)
        fills += op["n_fill"]
        ref = oracle.moe_ffn(list(bank_h[:E]), H, I, xb, oid, ow)
        assert_ffn_close(y.cpu().numpy(), ref, f"step {step}")
    _tables_equal(cache, ost)
    # every resident slot holds exactly its expert's bank blob
    pool = cache.pool.cpu().numpy()
    for slot, eid in enumerate(ost.id_of_slot):
        if eid >= 0:
            assert np.array_equal(pool[slot], bank_h[eid])
    assert fills > 0


@pytest.mark.parametrize("router,T,E", [("softmax", 16, 64), ("softmax", 17, 64),
                                          ("sigmoid_group", 16, 64), ("sigmoid_group", 17, 64),
                                          ("softmax", 3, 257)])
def test_layer_forward_selection_paths(oracle, router, T, E):
    """moe_layer_forward runs the router selection inside the control step for T <= 16 and
    E <= 256, with separate kernels otherwise: both give the oracle's ids, weights and plans."""
    H, I, k, S, K, L = 256, 128, 4, 24, 6, 2
    kw = dict(router="sigmoid_group", n_groups=8, topk_groups=3, routed_scale=2.5) \
        if router == "sigmoid_group" else {}
    spec = m.make_spec(L, H, I, E, k, **kw)
    bank_h = synth.make_bank(L * E, H, I, 5)
    bank = dev(bank_h, DEV)
    cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=bank, device=DEV)
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    ost = oracle.CacheState(L * E, S)
    for step in range(3):
        for layer in range(L):
            rng = np.random.default_rng(1000 * step + layer)
            xb = synth.bf16_bits(rng.normal(0, 1.5, (T, H)))
            wb = synth.router_weights(70 + layer, E, H)
            bias_h = synth.selection_bias(80 + layer, E) if router == "sigmoid_group" else None
            m.moe_layer_forward(spec, cache.c, layer, dev_bits(xb, DEV), T, dev_bits(wb, DEV),
                                None if bias_h is None else dev(bias_h, DEV), None, plan.c, ids,
                                wts, ws, wsb, y)
            torch.cuda.synchronize()
            ol = oracle.router_logits(xb, wb)
            if router == "sigmoid_group":
                oid, ow = oracle.route_sigmoid_group(ol, bias_h, 8, 3, k, 2.5)
            else:
                oid, ow = oracle.route_softmax_topk(ol, k)
            assert np.array_equal(ids.cpu().numpy(), oid)
            assert np.array_equal(f32_bits(wts.cpu().numpy()), f32_bits(ow))
            op = oracle.cache_step(ost, E, layer, oid, K, 52700, 77300)
            _plans_equal(plan.read(K), op, K)
    _tables_equal(cache, ost)


@pytest.mark.parametrize("H,I,E,k,T,shared", [(2048, 512, 256, 8, 1, True),
                                              (2048, 512, 256, 8, 8, True),
                                              (512, 192, 24, 3, 5, True),
                                              (7168, 2048, 16, 8, 1, False)])
def test_expert_ffn_direct_and_cached(oracle, H, I, E, k, T, shared):
    """FFN over a mix of hits, fills and direct (bank) experts, several tokens."""
    S = max(2, E // 4)
    spec, bank, bank_h, cache, sh = _layer_rig(1, H, I, E, k, S, 4, 11800, 47500, shared, seed=H)
    rng = np.random.default_rng(I)
    wr_h = synth.router_weights(I, E, H)
    wr = dev_bits(wr_h, DEV)
    plan = m.DevicePlan(T * k, 4, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    for step in range(3):
        xb = synth.bf16_bits(rng.normal(0, 2, (T, H)))
        m.moe_layer_forward(spec, cache.c, 0, dev_bits(xb, DEV), T, wr, None, sh, plan.c, ids,
                            wts, ws, wsb, y)
        torch.cuda.synchronize()
        gp = plan.read(4)
        oid, ow = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h), k)
        assert np.array_equal(ids.cpu().numpy(), oid)
        ref = oracle.moe_ffn(list(bank_h[:E]), H, I, xb, oid, ow,
                             bank_h[E] if shared else None, I)
        assert_ffn_close(y.cpu().numpy(), ref, f"step {step} plan {gp['counts']}")


def test_full_size_qwen_shape_decode(oracle):
    """40 layers x 256 experts (18.1 GB bank), 2560 slots, shared expert, T=1:
    four decode steps over all layers; layers 0, 17 and 39 checked against the oracle on
    every step, all 40 layers on the last step."""
    L, H, I, E, k, S, K, T = 40, 2048, 512, 256, 8, 2560, 8, 1
    spec, bank, _, cache, sh = _layer_rig(L, H, I, E, k, S, K, 52700, 77300, True, big=True)
    wr_h = [synth.router_weights(100 + l, E, H) for l in range(L)]
    wr = [dev_bits(w, DEV) for w in wr_h]
    xs = [synth.ar1_stream(l, 4, H) for l in range(L)]
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    ost = oracle.CacheState(L * E, S)
    shared_h = sh.cpu().numpy()
    for step in range(4):
        for layer in range(L):
            xb = xs[layer][step]
            m.moe_layer_forward(spec, cache.c, layer, dev_bits(xb, DEV), T, wr[layer], None, sh,
                                plan.c, ids, wts, ws, wsb, y)
            oid, ow = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h[layer]), k)
            op = oracle.cache_step(ost, E, layer, oid, K, 52700, 77300)
            if layer in (0, 17, 39) or step == 3:  # every layer on the last step
                torch.cuda.synchronize()
                assert np.array_equal(ids.cpu().numpy(), oid)
                _plans_equal(plan.read(K), op, K)
                blobs = {int(e): bank[layer * E + int(e)].cpu().numpy() for e in oid.reshape(-1)}
                full = [blobs.get(e, blobs[int(oid[0, 0])]) for e in range(E)]
                ref = oracle.moe_ffn(full, H, I, xb, oid, ow, shared_h, I)
                assert_ffn_close(y.cpu().numpy(), ref, f"step {step} layer {layer}")
    torch.cuda.synchronize()
    _tables_equal(cache, ost)
    # every resident slot holds its expert's blob, written by the FFN kernel that
    # carried the fill (compared on the device)
    assert m.moe_layer_kernel_count(spec, cache.c, T) == _layer_kernels(H, I, E, k, T, K, True)
    resident = [(v, int(e)) for v, e in enumerate(ost.id_of_slot) if e >= 0]
    assert resident
    for v, e in resident:
        assert torch.equal(cache.pool[v], bank[e]), f"slot {v} (id {e})"
    del bank, cache
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [1, 8])
def test_full_size_deepseek_shape_decode(oracle, T):
    """8 layers x 256 experts of H=7168, I=2048 (50.7 GB bank), sigmoid-group routing,
    307 slots, K=8, B_P/B_H = 11.8/47.5; sampled tokens checked against the oracle."""
    L, H, I, E, k, S, K = 8, 7168, 2048, 256, 8, 307, 8
    spec = m.make_spec(L, H, I, E, k, router="sigmoid_group", n_groups=8, topk_groups=4,
                       routed_scale=2.5)
    bank = synth.make_bank_torch(L * E, H, I, 7, DEV)
    cache = m.DeviceCache(spec, S, K, 11800, 47500, bank=bank, device=DEV)
    wr_h = [synth.router_weights(200 + l, E, H) for l in range(L)]
    bias_h = [synth.selection_bias(300 + l, E) for l in range(L)]
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    xs = [synth.ar1_stream(50 + l, 2, H, n_streams=T) for l in range(L)]
    ost = oracle.CacheState(L * E, S)
    for step in range(2):
        for layer in range(L):
            xb = xs[layer][step]
            m.moe_layer_forward(spec, cache.c, layer, dev_bits(xb, DEV), T,
                                dev_bits(wr_h[layer], DEV), dev(bias_h[layer], DEV), None,
                                plan.c, ids, wts, ws, wsb, y)
            ol = oracle.router_logits(xb, wr_h[layer])
            oid, ow = oracle.route_sigmoid_group(ol, bias_h[layer], 8, 4, k, 2.5)
            op = oracle.cache_step(ost, E, layer, oid, K, 11800, 47500)
            if layer in (0, 5) and step == 1:
                torch.cuda.synchronize()
                assert np.array_equal(ids.cpu().numpy(), oid)
                assert np.array_equal(f32_bits(wts.cpu().numpy()), f32_bits(ow))
                _plans_equal(plan.read(K), op, K)
                toks = [0] if T == 1 else [0, T - 1]
                need = {int(e) for t in toks for e in oid[t]}
                blobs = {e: bank[layer * E + e].cpu().numpy() for e in need}
                anyb = blobs[next(iter(need))]
                full = [blobs.get(e, anyb) for e in range(E)]
                ref = oracle.moe_ffn(full, H, I, xb[toks], oid[toks], ow[toks])
                assert_ffn_close(y.cpu().numpy()[toks], ref, f"layer {layer}")
    torch.cuda.synchronize()
    _tables_equal(cache, ost)
    # every resident slot holds its expert's blob, written by the FFN kernel that
    # carried the fill (compared on the device: 24.8 MB per slot)
    assert m.moe_layer_kernel_count(spec, cache.c, T) == _layer_kernels(H, I, E, k, T, K, True)
    resident = [(v, int(e)) for v, e in enumerate(ost.id_of_slot) if e >= 0]
    assert resident
    for v, e in resident:
        assert torch.equal(cache.pool[v], bank[e]), f"slot {v} (id {e})"
    del bank, cache
    torch.cuda.empty_cache()


@pytest.mark.parametrize("H,I,T", [(1024, 256, 4), (1024, 512, 6), (1536, 128, 3), (512, 192, 12)])
def test_expert_ffn_repeated_ids(oracle, H, I, T):
    """Routing given by the caller in which one token lists an expert twice and
    several tokens share experts: each (token, rank) pair contributes once."""
    E, k = 8, 3
    spec, bank, bank_h, cache, _ = _layer_rig(1, H, I, E, k, 2, 2, 11800, 47500, False, seed=I)
    rng = np.random.default_rng(H + T)
    ids_h = rng.integers(0, E, (T, k)).astype(np.int32)
    ids_h[0] = [5, 5, 2]
    ids_h[1, 0] = 5
    w_h = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    xb = synth.bf16_bits(rng.normal(0, 1, (T, H)))
    plan = m.DevicePlan(T * k, 2, device=DEV)
    fws = m.moe_ffn_workspace_bytes(spec, T)
    ws = torch.empty(fws, dtype=torch.uint8, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    ids = dev(ids_h, DEV)
    for step in range(2):  # second pass runs with the slots filled by the first
        m.moe_cache_step(spec, cache.c, 0, ids, T, plan.c, 1)
        m.moe_expert_ffn(spec, cache.c, 0, plan.c, dev_bits(xb, DEV), T, ids, dev(w_h, DEV), None,
                         ws, fws, y)
        torch.cuda.synchronize()
        assert plan.read(2)["err"] == 0
        ref = oracle.moe_ffn(list(bank_h[:E]), H, I, xb, ids_h, w_h)
        assert_ffn_close(y.cpu().numpy(), ref, f"step {step}")


@pytest.mark.parametrize("H,I", [(1024, 256), (256, 128), (1024, 512)])
def test_expert_ffn_no_valid_expert_writes_zero(oracle, H, I):
    """Every routed id out of range and no shared expert: the control step flags
    the ids, nothing executes, and y is all zeros (stale contents are replaced)."""
    E, k, T = 8, 2, 1
    spec, bank, bank_h, cache, _ = _layer_rig(1, H, I, E, k, 2, 2, 11800, 47500, False, seed=3)
    plan = m.DevicePlan(T * k, 2, device=DEV)
    fws = m.moe_ffn_workspace_bytes(spec, T)
    ws = torch.empty(fws, dtype=torch.uint8, device=DEV)
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    ids = torch.tensor([[E, -1]], dtype=torch.int32, device=DEV)
    w = torch.tensor([[0.5, 0.5]], dtype=torch.float32, device=DEV)
    xb = synth.bf16_bits(np.random.default_rng(0).normal(0, 1, (T, H)))
    m.moe_cache_step(spec, cache.c, 0, ids, T, plan.c, 1)
    m.moe_expert_ffn(spec, cache.c, 0, plan.c, dev_bits(xb, DEV), T, ids, w, None, ws, fws, y)
    torch.cuda.synchronize()
    gp = plan.read(2)
    assert gp["err"] & m.MOE_DERR_BAD_ID and gp["n_uniq"] == 0
    assert torch.count_nonzero(y).item() == 0


def test_profile_bandwidths_leaves_cache_and_feeds_q(oracle):
    """On-device B_P / B_H: positive rates, the cache (tables, stamps, clock, slot pool)
    untouched, and a control step with the measured values still matches the oracle."""
    L, H, I, E, k, S, K = 2, 2048, 512, 16, 8, 6, 8
    spec, bank, bank_h, cache, _ = _layer_rig(L, H, I, E, k, S, K, 52700, 77300, False)
    plan = m.DevicePlan(k, K, device=DEV)
    ost = oracle.CacheState(L * E, S)
    rng = np.random.default_rng(11)
    for step in range(4):  # populate some slots
        ids_h = rng.choice(E, size=(1, k), replace=False).astype(np.int32)
        m.moe_cache_step(spec, cache.c, step % L, dev(ids_h, DEV), 1, plan.c, 1)
        oracle.cache_step(ost, E, step % L, ids_h, K, 52700, 77300)
    torch.cuda.synchronize()
    before = cache.host_tables()
    pool_before = cache.pool.clone()
    wsb = m.moe_profile_workspace_bytes(spec)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    bp, bh = m.moe_profile_bandwidths(spec, cache.c, 1, ws, wsb, reps=4)
    assert 1_000 < bp < 100_000_000 and 1_000 < bh < 100_000_000, (bp, bh)
    after = cache.host_tables()
    for x, y in zip(before, after):
        assert np.array_equal(x, y)
    assert torch.equal(pool_before, cache.pool)
    # the measured rates drive q* like configured ones
    cache.c.bp_mbps, cache.c.bh_mbps = bp, bh
    ids_h = rng.choice(E, size=(1, k), replace=False).astype(np.int32)
    m.moe_cache_step(spec, cache.c, 0, dev(ids_h, DEV), 1, plan.c, 0)
    torch.cuda.synchronize()
    op = oracle.cache_step(ost, E, 0, ids_h, K, bp, bh)
    _plans_equal(plan.read(K), op, K)
