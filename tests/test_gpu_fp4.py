"""GPU parity of the FP4 decode path (MXFP4, NVFP4: the formats of the pages'
deployed models, FreeToken summary "Key results" table) against the CPU
oracle's FP4 expert (or_fp4_expert_forward), through the C ABI.

The layer output is the routed experts' outputs weighted by the routing
weights plus the shared expert's, summed here in float64 from the oracle's
per-expert results; outputs must be within the Edge0 tolerance (relative L2
<= 1e-2, |err| <= 2e-2 * max|y|).  Routing, plans and slot tables are format-
independent and must match bit for bit; every resident slot must hold its
bank blob byte for byte.
"""
import numpy as np
import pytest

import moe_expert_offload_gb300 as m
from moe_expert_offload_gb300 import synth

from gpu_util import assert_ffn_close, dev, dev_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"
# ABI format -> the oracle's FP4 format number (0 MXFP4, 1 NVFP4)
ORACLE_FMT = {m.FORMAT_MXFP4: 0, m.FORMAT_NVFP4: 1}


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


def _fp4_bank(n, H, I, fmt, seed):
    rng = np.random.default_rng(seed)
    return np.stack([synth.make_fp4_expert(rng, H, I, ORACLE_FMT[fmt]) for _ in range(n)])


def _reference(oracle, blobs, H, I, fmt, xb, ids, wts, shared_blob=None):
    """y[t] = sum_j w[t][j] expert_{ids[t][j]}(x[t]) (+ shared(x[t])), float64; each
    expert's output is the oracle's FP4 forward over all tokens at once."""
    T = xb.shape[0]
    y = np.zeros((T, H), dtype=np.float64)
    of = ORACLE_FMT[fmt]
    cache = {}
    for e in np.unique(ids):
        cache[int(e)] = oracle.fp4_expert_forward(blobs[int(e)], H, I, of, xb)
    for t in range(T):
        for j in range(ids.shape[1]):
            y[t] += float(wts[t, j]) * cache[int(ids[t, j])][t]
    if shared_blob is not None:
        y += oracle.fp4_expert_forward(shared_blob, H, I, of, xb)
    return y


def test_fp4_blob_bytes_match_the_oracle_layout(oracle):
    for fmt in (m.FORMAT_MXFP4, m.FORMAT_NVFP4):
        for H, I in ((1024, 512), (2048, 512), (7168, 2048)):
            spec = m.make_spec(1, H, I, 8, 2, fmt=fmt)
            assert m.moe_expert_bytes(spec) == oracle.fp4_blob_offsets(H, I, ORACLE_FMT[fmt])[
                "total"]


@pytest.mark.parametrize("fmt", [m.FORMAT_MXFP4, m.FORMAT_NVFP4])
@pytest.mark.parametrize("H,I,E,k,T,shared", [(1024, 512, 16, 4, 1, True),
                                              (2048, 512, 16, 8, 4, False),
                                              (2048, 1024, 12, 4, 8, True),
                                              (3072, 512, 20, 6, 5, True)])
def test_fp4_expert_ffn_matches_oracle(oracle, fmt, H, I, E, k, T, shared):
    """moe_expert_ffn on FP4 experts: some resident in slots, the rest read from
    the bank; the routed ids include repeats across tokens.  Both down-tile
    geometries (inter % 1024 == 0 or not) and 1..8 tokens."""
    bank_h = _fp4_bank(E + 1, H, I, fmt, seed=H + T + fmt)
    bank = dev(bank_h, DEV)
    spec = m.make_spec(1, H, I, E, k, has_shared=shared, fmt=fmt)
    assert m.moe_expert_bytes(spec) == bank_h.shape[1]
    S, K = max(2, E // 3), 2
    cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=bank[:E], device=DEV)
    m.moe_cache_place(spec, cache.c, list(range(0, E, 3))[:S])
    plan = m.DevicePlan(T * k, K, device=DEV)
    rng = np.random.default_rng(T)
    ids_h = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    wts_h = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    xb = synth.bf16_bits(rng.normal(0, 1.5, (T, H)))
    ids, wts = dev(ids_h, DEV), dev(wts_h, DEV)
    sh = bank[E] if shared else None
    # the step's plan (hits, fills, direct); the fill runs as a copy kernel here
    m.moe_cache_step(spec, cache.c, 0, ids, T, plan.c, 1)
    ws_b = m.moe_ffn_workspace_bytes(spec, T)
    ws = torch.empty(ws_b, dtype=torch.uint8, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    m.moe_expert_ffn(spec, cache.c, 0, plan.c, dev_bits(xb, DEV), T, ids, wts, sh, ws, ws_b, y)
    torch.cuda.synchronize()
    assert int(plan.err[0].item()) == 0
    ref = _reference(oracle, bank_h, H, I, fmt, xb, ids_h, wts_h, bank_h[E] if shared else None)
    assert_ffn_close(y.cpu().numpy(), ref, f"fmt {fmt} H {H} I {I} T {T}")


@pytest.mark.parametrize("fmt", [m.FORMAT_MXFP4, m.FORMAT_NVFP4])
@pytest.mark.parametrize("sync", [True, False])
def test_fp4_layer_forward_matches_oracle(oracle, fmt, sync):
    """moe_layer_forward on FP4 experts over 10 steps with fills and evictions:
    routing and plans bit for bit, outputs within tolerance, every resident slot
    byte-equal to its bank blob (the fill written by the FFN kernel).  With the
    cache's sync words the step is one kernel."""
    L, H, I, E, k, T, S, K = 2, 1024, 512, 16, 4, 2, 6, 3
    bank_h = _fp4_bank(L * E + 1, H, I, fmt, seed=7 + fmt)
    bank = dev(bank_h, DEV)
    spec = m.make_spec(L, H, I, E, k, has_shared=True, fmt=fmt)
    cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=bank[:L * E], device=DEV, sync=sync)
    assert m.moe_layer_kernel_count(spec, cache.c, T) == (1 if sync else 3)
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    ost = oracle.CacheState(L * E, S)
    rng = np.random.default_rng(11)
    fills = 0
    for step in range(10):
        layer = step % L
        wr_h = synth.router_weights(60 + layer, E, H)
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
        fills += op["n_fill"]
        ref = _reference(oracle, bank_h[layer * E:(layer + 1) * E], H, I, fmt, xb, oid, ow,
                         bank_h[L * E])
        assert_ffn_close(y.cpu().numpy(), ref, f"step {step}")
        pool = cache.pool.cpu().numpy()
        for slot, eid in enumerate(ost.id_of_slot):
            if eid >= 0:
                assert np.array_equal(pool[slot], bank_h[eid]), f"step {step} slot {slot}"
    assert fills > 0
    assert int(plan.err[0].item()) == 0


@pytest.mark.parametrize("fmt", [m.FORMAT_MXFP4, m.FORMAT_NVFP4])
def test_fp4_qwen_shape_layer_steps(oracle, fmt):
    """Qwen3.6-shaped FP4 layer (H=2048, I=512, E=256, top-8 + shared expert), 4
    layers, 3 decode steps through the one-kernel step; every layer's output
    checked on the last step, slot bytes equal to the bank's."""
    L, H, I, E, k, S, K, T = 4, 2048, 512, 256, 8, 256, 8, 1
    of = ORACLE_FMT[fmt]
    bank = synth.make_fp4_bank_torch(L * E + 1, H, I, of, 21 + fmt, DEV)
    spec = m.make_spec(L, H, I, E, k, has_shared=True, fmt=fmt)
    cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=bank[:L * E], device=DEV)
    assert m.moe_layer_kernel_count(spec, cache.c, T) == 1
    wr_h = [synth.router_weights(300 + l, E, H) for l in range(L)]
    xs = [synth.ar1_stream(40 + l, 3, H) for l in range(L)]
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    shared_h = bank[L * E].cpu().numpy()
    for step in range(3):
        for layer in range(L):
            xb = xs[layer][step]
            m.moe_layer_forward(spec, cache.c, layer, dev_bits(xb, DEV), T,
                                dev_bits(wr_h[layer], DEV), None, bank[L * E], plan.c, ids, wts,
                                ws, wsb, y)
            if step == 2:
                torch.cuda.synchronize()
                oid, ow = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h[layer]), k)
                assert np.array_equal(ids.cpu().numpy(), oid)
                blobs = {int(e): bank[layer * E + int(e)].cpu().numpy() for e in oid.reshape(-1)}
                ref = _reference(oracle, blobs, H, I, fmt, xb, oid, ow, shared_h)
                assert_ffn_close(y.cpu().numpy(), ref, f"layer {layer}")
    torch.cuda.synchronize()
    assert int(plan.err[0].item()) == 0
    ids_of = cache.id_of_slot.cpu().numpy()
    for v in np.nonzero(ids_of >= 0)[0][:64]:
        assert torch.equal(cache.pool[v], bank[int(ids_of[v])]), f"slot {v}"


# ------------------------------------------------------------------ prefill
def _prefill_reference(oracle, blobs, H, I, fmt, xb, ids, wts, shared_blob=None):
    """y[t] = sum_j w[t][j] expert_{ids[t][j]}(x[t]) (+ shared(x[t])), float64; each
    expert's oracle FP4 forward runs on the rows routed to it only."""
    T = xb.shape[0]
    of = ORACLE_FMT[fmt]
    y = np.zeros((T, H), dtype=np.float64)
    for e in np.unique(ids):
        rows = np.nonzero((ids == e).any(axis=1))[0]
        ye = oracle.fp4_expert_forward(blobs[int(e)], H, I, of, xb[rows])
        for n, t in enumerate(rows):
            y[t] += float(wts[t][ids[t] == e].sum()) * ye[n]
    if shared_blob is not None:
        y += oracle.fp4_expert_forward(shared_blob, H, I, of, xb)
    return y


def _prefill(spec, experts, shared, xb, ids_h, w_h):
    T, H = xb.shape[0], spec.hidden
    wsb = m.moe_prefill_workspace_bytes(spec, T)
    assert wsb > 0
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    m.moe_expert_ffn_prefill(spec, experts, dev_bits(xb, DEV), T, dev(ids_h, DEV), dev(w_h, DEV),
                             shared, err, ws, wsb, y)
    torch.cuda.synchronize()
    assert int(err.cpu()[0]) == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("fmt", [m.FORMAT_MXFP4, m.FORMAT_NVFP4])
@pytest.mark.parametrize("H,I,E,k,T,shared", [(256, 128, 16, 2, 300, True),
                                              (1024, 256, 32, 4, 400, False),
                                              (2048, 512, 16, 4, 200, True)])
def test_fp4_prefill_matches_oracle(oracle, fmt, H, I, E, k, T, shared):
    """moe_expert_ffn_prefill on FP4 experts (the grouped tcgen05 GEMMs with the
    weights dequantised to bf16 in the kernel) against the oracle's FP4 expert."""
    spec = m.make_spec(1, H, I, E, k, has_shared=shared, fmt=fmt)
    bank_h = _fp4_bank(E + 1, H, I, fmt, seed=H + T + 10 * fmt)
    bank = dev(bank_h, DEV)
    rng = np.random.default_rng(T + fmt)
    xb = synth.bf16_bits(rng.normal(0, 1.5, (T, H)))
    wr_h = synth.router_weights(E, E, H)
    ids_h, w_h = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h), k)
    y = _prefill(spec, bank[:E], bank[E] if shared else None, xb, ids_h, w_h)
    ref = _prefill_reference(oracle, bank_h, H, I, fmt, xb, ids_h, w_h,
                             bank_h[E] if shared else None)
    assert_ffn_close(y, ref, f"fp4 prefill fmt {fmt} H {H} T {T}")


@pytest.mark.parametrize("fmt", [m.FORMAT_MXFP4, m.FORMAT_NVFP4])
def test_fp4_prefill_wide_scales_and_multi_tile_experts(oracle, fmt):
    """Block scales across a wide range (MXFP4 E8M0 bytes 100..150, i.e. 2^-27 ..
    2^23, beyond what the decode kernel's fp16 products hold; NVFP4 E4M3 bytes
    including subnormals and the largest finite value 448), and skewed routing:
    two experts take most rows, so each spans several 256-row m-tiles."""
    H, I, E, k, T = 256, 128, 8, 2, 700
    of = ORACLE_FMT[fmt]
    spec = m.make_spec(1, H, I, E, k, has_shared=False, fmt=fmt)
    bank_h = _fp4_bank(E, H, I, fmt, seed=99 + fmt)
    off = oracle.fp4_blob_offsets(H, I, of)
    rng = np.random.default_rng(5 + fmt)
    n_sc = off["mat"] - off["gs"]
    if fmt == m.FORMAT_MXFP4:
        bank_h[:, off["gs"]:off["mat"]] = rng.integers(100, 151, size=(E, n_sc), dtype=np.uint8)
    else:
        sc = rng.integers(0, 0x7F, size=(E, n_sc), dtype=np.uint8)  # no NaN (0x7F)
        sc[:, ::17] = 0x7E                                           # 448
        sc[:, 3::29] = rng.integers(1, 8, size=sc[:, 3::29].shape)  # subnormals
        bank_h[:, off["gs"]:off["mat"]] = sc
    bank = dev(bank_h, DEV)
    xb = synth.bf16_bits(rng.normal(0, 1, (T, H)))
    ids_h = np.zeros((T, k), np.int32)
    ids_h[:, 0] = 3
    ids_h[:, 1] = np.where(rng.random(T) < 0.9, 6, rng.integers(0, 3, T))
    w_h = np.tile(np.array([[0.7, 0.3]], np.float32), (T, 1))
    y = _prefill(spec, bank, None, xb, ids_h, w_h)
    ref = _prefill_reference(oracle, bank_h, H, I, fmt, xb, ids_h, w_h)
    assert_ffn_close(y, ref, f"fp4 prefill wide scales fmt {fmt}")


def test_fp4_full_size_prefill_layer(oracle):
    """The qwen_prefill_nvfp4 shape: one Qwen-shaped NVFP4 layer, 8192 tokens whose
    routing union covers all 256 experts, through moe_layer_forward_prefill.  Against
    the oracle's FP4 expert: 64 rows spread over the m-tiles of the two experts with
    the most assignments (each spans several 256-row m-tiles) and 16 rows of the
    shared expert's group."""
    H, I, E, k, T = 2048, 512, 256, 8, 8192
    fmt = m.FORMAT_NVFP4
    spec = m.make_spec(1, H, I, E, k, has_shared=True, fmt=fmt)
    bank = synth.make_fp4_bank_torch(E + 1, H, I, ORACLE_FMT[fmt], 13, DEV)
    wr_h = synth.router_weights(78, E, H)
    xb = synth.prefill_hidden(4, T, H, wr_h)
    wsb = m.moe_prefill_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    m.moe_layer_forward_prefill(spec, bank[:E], dev_bits(xb, DEV), T, dev_bits(wr_h, DEV), None,
                                bank[E], ids, wts, err, ws, wsb, y)
    torch.cuda.synchronize()
    assert int(err.cpu()[0]) == 0
    ids_g, w_g, y_g = ids.cpu().numpy(), wts.cpu().numpy(), y.cpu().numpy()
    assert len(np.unique(ids_g)) == E
    assert np.all(np.isfinite(y_g))
    counts = np.bincount(ids_g.reshape(-1), minlength=E)
    top2 = np.argsort(-counts, kind="stable")[:2]
    assert counts[top2].min() > 256, counts[top2]
    rows = set()
    for e in top2:
        r = np.nonzero((ids_g == e).any(axis=1))[0]
        rows |= set(r[np.linspace(0, len(r) - 1, 32).round().astype(int)].tolist())
    rows |= set(range(4096, 4096 + 256, 16))
    rows = np.asarray(sorted(rows))
    blobs = {int(e): bank[int(e)].cpu().numpy() for e in np.unique(ids_g[rows])}
    ref = _prefill_reference(oracle, blobs, H, I, fmt, xb[rows], ids_g[rows], w_g[rows],
                             bank[E].cpu().numpy())
    assert_ffn_close(y_g[rows], ref, f"full-size NVFP4 prefill: {len(rows)} rows")
    del bank
    torch.cuda.empty_cache()
