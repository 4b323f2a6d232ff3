"""GPU parity of the prefill path (routing permute, tcgen05 grouped GEMMs,
combine, whole-layer copy) against the CPU oracle, through the C ABI.

The prefill FFN rounds h and each weighted expert output to bf16 (the GEMM
operand and the combine's input); the Edge0 tolerance still applies:
relative L2 <= 1e-2 and |err| <= 2e-2 * max|y|."""
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


def _run_prefill(spec, experts, shared, xb, ids_h, w_h):
    T = xb.shape[0]
    H = spec.hidden
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


@pytest.mark.parametrize("H,I,E,k,T,shared", [(256, 128, 16, 2, 300, True),
                                              (256, 128, 16, 2, 1, False),
                                              (512, 256, 64, 4, 1000, True),
                                              (2048, 512, 32, 8, 700, True)])
def test_prefill_ffn_matches_oracle(oracle, H, I, E, k, T, shared):
    spec = m.make_spec(1, H, I, E, k, has_shared=shared)
    bank_h = synth.make_bank(E + 1, H, I, seed=H + T)
    bank = dev(bank_h, DEV)
    rng = np.random.default_rng(T)
    xb = synth.bf16_bits(rng.normal(0, 1.5, (T, H)))
    wr_h = synth.router_weights(E, E, H)
    ids_h, w_h = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h), k)
    y = _run_prefill(spec, bank[:E], bank[E] if shared else None, xb, ids_h, w_h)
    ref = oracle.moe_ffn(list(bank_h[:E]), H, I, xb, ids_h, w_h,
                         bank_h[E] if shared else None, I)
    assert_ffn_close(y, ref, f"prefill H={H} E={E} T={T}")


def test_prefill_skewed_routing_and_empty_experts(oracle):
    # most tokens on two experts (tiles of many rows), several experts unused
    H, I, E, k, T = 256, 128, 16, 2, 513
    spec = m.make_spec(1, H, I, E, k, has_shared=False)
    bank_h = synth.make_bank(E, H, I, seed=5)
    bank = dev(bank_h, DEV)
    rng = np.random.default_rng(9)
    xb = synth.bf16_bits(rng.normal(0, 1, (T, H)))
    ids_h = np.zeros((T, k), np.int32)
    ids_h[:, 0] = 3
    ids_h[:, 1] = np.where(rng.random(T) < 0.9, 11, rng.integers(0, 3, T))
    w_h = np.tile(np.array([[0.75, 0.25]], np.float32), (T, 1))
    y = _run_prefill(spec, bank, None, xb, ids_h, w_h)
    ref = oracle.moe_ffn(list(bank_h), H, I, xb, ids_h, w_h)
    assert_ffn_close(y, ref, "skewed")


@pytest.mark.parametrize("offset", [0, 16, 4])
def test_layer_prefetch_copies_the_layer(offset):
    """The layer copy lands byte for byte and writes nothing around dst: the
    copy kernel at 16-byte aligned destinations, the plain copy at offset 4."""
    H, I, E, L = 256, 128, 16, 3
    spec = m.make_spec(L, H, I, E, 2)
    se = m.moe_expert_bytes(spec)
    bank = dev(synth.make_bank(L * E, H, I, seed=2), DEV)
    buf = torch.zeros(E * se + 64, dtype=torch.uint8, device=DEV)
    dst = buf[offset:offset + E * se]
    side = torch.cuda.Stream()
    m.moe_layer_prefetch(spec, bank, 2, dst, side)
    side.synchronize()
    assert torch.equal(dst, bank[2 * E:3 * E].reshape(-1))
    assert not buf[:offset].any() and not buf[offset + E * se:].any()


def test_layer_prefetch_beside_routing_full_layer():
    """A whole Qwen-shaped layer (256 experts, 453 MB) copied on a second stream
    while moe_route runs on the first: the copy is exact and the routing equals
    the routing run alone."""
    L, H, I, E, k, T = 2, 2048, 512, 256, 8, 4096
    spec = m.make_spec(L, H, I, E, k)
    se = m.moe_expert_bytes(spec)
    bank = torch.randint(0, 256, (L * E, se), dtype=torch.uint8, device=DEV)
    dst = torch.empty((E, se), dtype=torch.uint8, device=DEV)
    rng = np.random.default_rng(11)
    xb = torch.from_numpy(synth.bf16_bits(rng.normal(0, 1, (T, H))).view(np.int16)).to(DEV)
    wr = torch.from_numpy(synth.router_weights(3, E, H).view(np.int16)).to(DEV)

    def route(stream):
        logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
        ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
        wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
        m.moe_route(spec, xb, T, wr, None, logits, ids, wts, stream.cuda_stream)
        return logits, ids, wts

    main = torch.cuda.current_stream()
    want = route(main)
    torch.cuda.synchronize()
    side = torch.cuda.Stream(priority=-1)
    m.moe_layer_prefetch(spec, bank, 1, dst, side.cuda_stream)
    got = route(main)
    torch.cuda.synchronize()
    assert torch.equal(dst, bank[E:2 * E])
    for a, b in zip(got, want):
        assert torch.equal(a, b)


def test_full_size_qwen_prefill_layer(oracle):
    """One Qwen-shaped layer, 8192 tokens with router logits raised on expert t mod 256 so the
    routing union covers all 256 experts; routing on sampled tokens bit-exact; against the
    oracle, every output row of the two experts with the most assignments (several m-tiles
    each) and a full 256-row m-tile of the shared expert."""
    H, I, E, k, T = 2048, 512, 256, 8, 8192
    spec = m.make_spec(1, H, I, E, k, has_shared=True)
    bank = synth.make_bank_torch(E + 1, H, I, 11, DEV)
    wr_h = synth.router_weights(77, E, H)
    xb = synth.prefill_hidden(3, T, H, wr_h)
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
    assert len(np.unique(ids_g)) == E  # the union covers every expert
    sample = np.random.default_rng(0).choice(T, 48, replace=False)
    lg = oracle.router_logits(xb[sample], wr_h)
    oid, ow = oracle.route_softmax_topk(lg, k)
    assert np.array_equal(ids_g[sample], oid)
    assert np.array_equal(f32_bits(w_g[sample]), f32_bits(ow))
    # every output row of the two experts with the most assignments (each spans two or more
    # 256-row m-tiles of its group), and one full 256-row m-tile of the shared expert's group
    # (the shared group takes the tokens in order)
    counts = np.bincount(ids_g.reshape(-1), minlength=E)
    top2 = np.argsort(-counts, kind="stable")[:2]
    assert counts[top2].min() > 256, counts[top2]
    rows = sorted(set(np.nonzero(np.isin(ids_g, top2).any(axis=1))[0].tolist()) |
                  set(range(2048, 2048 + 256)))
    rows = np.asarray(rows)
    blobs = list(bank[:E].cpu().numpy())
    import os
    oracle.set_threads(os.cpu_count() or 1)
    try:
        ref = oracle.moe_ffn(blobs, H, I, xb[rows], ids_g[rows], w_g[rows],
                             bank[E].cpu().numpy(), I)
    finally:
        oracle.set_threads(1)
    assert_ffn_close(y_g[rows], ref, f"full-size prefill: {len(rows)} rows")
    assert np.all(np.isfinite(y_g))
    del bank
    torch.cuda.empty_cache()
