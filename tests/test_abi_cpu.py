"""Host-side checks of the C-ABI library: it loads without a GPU, exports every
function the public headers declare, and rejects bad arguments on the host
(before any CUDA call) with the documented status codes."""
import ctypes as C
import glob
import os
import re

import pytest

import moe_expert_offload_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \t\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    from moe_expert_offload_gb300 import _build

    _build.build()
    return m.lib()


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert "moe_route" in declared and "moe_layer_forward" in declared
    for name in declared:
        assert hasattr(L, name), f"libmoe.so does not export {name}"
    assert set(m.EXPORTED) <= set(declared)


def test_version_and_error_string(L):
    assert "sm_103a" in m.moe_version()
    assert isinstance(m.moe_last_error(), str)


def _spec(**kw):
    base = dict(num_layers=2, hidden=256, inter=128, num_experts=16, top_k=2)
    base.update(kw)
    return m.make_spec(**base)


def test_expert_bytes_matches_layout(L):
    assert m.moe_expert_bytes(_spec()) == 55_296
    assert m.moe_expert_bytes(_spec(hidden=2048, inter=512, num_experts=256, top_k=8)) == 1_769_472
    assert m.moe_expert_bytes(_spec(hidden=7168, inter=2048, num_experts=256, top_k=8)) == 24_772_608


def test_fp4_expert_bytes_match_the_oracle_layout(L):
    """The library's FP4 blob size agrees with the oracle's own layout (two
    separate implementations of the same reading)."""
    import oracle

    oracle.build()
    for fmt, ofmt in ((m.FORMAT_MXFP4, oracle.MXFP4), (m.FORMAT_NVFP4, oracle.NVFP4)):
        for H, I in ((256, 128), (2048, 512), (7168, 2048), (1024, 192)):
            got = m.moe_expert_bytes(_spec(hidden=H, inter=I, fmt=fmt))
            assert got == oracle.fp4_blob_offsets(H, I, ofmt)["total"], (fmt, H, I)


def test_fp4_prefill_workspace_is_format_independent(L):
    """The prefill path takes FP4 experts (dequantised to bf16 in the GEMM); its
    scratch (permute, h, weighted outputs) does not depend on the weight format."""
    for T in (1, 300, 8192):
        want = m.moe_prefill_workspace_bytes(_spec(hidden=1024, inter=512), T)
        assert want > 0
        for fmt in (m.FORMAT_MXFP4, m.FORMAT_NVFP4):
            assert m.moe_prefill_workspace_bytes(_spec(hidden=1024, inter=512, fmt=fmt), T) == want


@pytest.mark.parametrize("kw", [
    dict(fmt=3), dict(fmt=-1),
    dict(hidden=100), dict(inter=96), dict(num_experts=0), dict(num_experts=2000),
    dict(top_k=0), dict(top_k=17), dict(num_layers=0),
    dict(router="sigmoid_group", n_groups=3), dict(router="sigmoid_group", n_groups=4, topk_groups=5),
    dict(router="sigmoid_group", n_groups=16, topk_groups=1, top_k=2),
])
def test_bad_spec_rejected(L, kw):
    s = _spec(**kw)
    assert m.moe_expert_bytes(s) == 0
    with pytest.raises(m.MoeError) as e:
        m.moe_route(s, 16, 1, 16, None, 16, 16, 16, stream=0)
    assert e.value.code in (m.MOE_EINVAL, m.MOE_EUNSUPPORTED)


def test_unsupported_group_size(L):
    s = _spec()
    s.group_size = 32
    with pytest.raises(m.MoeError) as e:
        m.moe_route(s, 16, 1, 16, None, 16, 16, 16, stream=0)
    assert e.value.code == m.MOE_EUNSUPPORTED


def test_route_argument_checks(L):
    s = _spec()
    with pytest.raises(m.MoeError) as e:
        m.moe_route(s, 16, -1, 16, None, 16, 16, 16, stream=0)
    assert e.value.code == m.MOE_EINVAL
    with pytest.raises(m.MoeError) as e:
        m.moe_route(s, None, 1, 16, None, 16, 16, 16, stream=0)
    assert e.value.code == m.MOE_EINVAL
    with pytest.raises(m.MoeError) as e:
        m.moe_route(s, 18, 1, 16, None, 16, 16, 16, stream=0)  # misaligned x
    assert e.value.code == m.MOE_EINVAL
    assert m.moe_route(s, None, 0, None, None, None, None, None, stream=0) == m.MOE_OK


def _cache(**kw):
    c = dict(num_slots=8, k_victims=4, bp_mbps=52700, bh_mbps=77300, slot_of_id=256,
             id_of_slot=512, ts=768, clock=1024, slot_pool=4096, bank=8192)
    c.update(kw)
    return m.MoeCache(**c)


def _plan(cap=2):
    return m.MoePlan(cap, *([256] * 10))


@pytest.mark.parametrize("kw,code", [
    (dict(num_slots=0), m.MOE_EINVAL), (dict(k_victims=0), m.MOE_EINVAL),
    (dict(k_victims=33), m.MOE_EINVAL), (dict(bp_mbps=0), m.MOE_EINVAL),
    (dict(ts=None), m.MOE_EINVAL), (dict(bank=None), m.MOE_EINVAL),
    (dict(slot_pool=4100), m.MOE_EINVAL), (dict(policy=3), m.MOE_EINVAL),
    (dict(policy=-1), m.MOE_EINVAL), (dict(policy=m.POLICY_LAYER_LRU, num_slots=1), m.MOE_EINVAL),
])
def test_cache_step_rejects_bad_cache(L, kw, code):
    with pytest.raises(m.MoeError) as e:
        m.moe_cache_step(_spec(), _cache(**kw), 0, 64, 1, _plan(), 1, stream=0)
    assert e.value.code == code


def test_cache_step_rejects_bad_layer_and_capacity(L):
    with pytest.raises(m.MoeError) as e:
        m.moe_cache_step(_spec(), _cache(), 2, 64, 1, _plan(), 1, stream=0)
    assert e.value.code == m.MOE_EINVAL
    with pytest.raises(m.MoeError) as e:
        m.moe_cache_step(_spec(), _cache(), 0, 64, 2, _plan(cap=3), 1, stream=0)
    assert e.value.code == m.MOE_ECAPACITY
    with pytest.raises(m.MoeError) as e:
        m.moe_cache_step(_spec(), _cache(), 0, 64, 513, _plan(cap=2000), 1, stream=0)
    assert e.value.code == m.MOE_ECAPACITY
    p = _plan()
    p.err = None
    with pytest.raises(m.MoeError) as e:
        m.moe_cache_step(_spec(), _cache(), 0, 64, 1, p, 1, stream=0)
    assert e.value.code == m.MOE_EINVAL
    assert m.moe_cache_step(_spec(), _cache(), 0, 64, 0, _plan(), 1, stream=0) == m.MOE_OK


def test_cache_place_argument_checks(L):
    # every rejection happens on the host before any device write
    sp = _spec()
    E, nl = sp.num_experts, sp.num_layers
    bad = [([3, 3], m.POLICY_SHARED_LRU), ([nl * E], m.POLICY_SHARED_LRU),
           ([-1], m.POLICY_STATIC), (list(range(9)), m.POLICY_SHARED_LRU),
           ([0, 1, 2, 3, 4], m.POLICY_LAYER_LRU)]  # dup, range, range, > S, > S_l = 4
    for ids, pol in bad:
        with pytest.raises(m.MoeError) as e:
            m.moe_cache_place(sp, _cache(policy=pol), ids, stream=0)
        assert e.value.code == m.MOE_EINVAL, (ids, pol)
    with pytest.raises(m.MoeError) as e:
        m.moe_cache_place(sp, _cache(policy=5), [1], stream=0)
    assert e.value.code == m.MOE_EINVAL
    with pytest.raises(m.MoeError) as e:
        m._check(L.moe_cache_place(C.byref(sp), C.byref(_cache()), None, 2, None))
    assert e.value.code == m.MOE_EINVAL


def test_slots_for_budget_and_resize_workspace(L):
    """floor(free / S_e) with the library's own blob size (the oracle's
    restatement is pinned to the reader's 10 / 8 / 12 example)."""
    import oracle

    oracle.build()
    for kw in (dict(), dict(hidden=2048, inter=512, num_experts=256, top_k=8),
               dict(hidden=1024, inter=512, fmt=m.FORMAT_NVFP4)):
        sp = _spec(**kw)
        se = m.moe_expert_bytes(sp)
        for free in (0, se - 1, se, 5 << 30, 4 << 30, 6 << 30):
            assert m.moe_slots_for_budget(sp, free) == oracle.slots_for_budget(free, se)
    with pytest.raises(m.MoeError):
        m.moe_slots_for_budget(_spec(), -1)
    with pytest.raises(m.MoeError):
        m.moe_slots_for_budget(_spec(num_layers=0), 1 << 20)
    c = _cache(num_slots=10)
    assert m.moe_cache_resize_workspace_bytes(c, 8) == 4 * (8 + 3 * 10)
    assert m.moe_cache_resize_workspace_bytes(c, 12) == 4 * (8 + 3 * 12)
    assert m.moe_cache_resize_workspace_bytes(c, 0) == 0


def test_cache_resize_argument_checks(L):
    sp = _spec()
    need = m.moe_cache_resize_workspace_bytes(_cache(), 4)
    cases = [(_cache(policy=m.POLICY_LAYER_LRU), 4, 4096, need, m.MOE_EUNSUPPORTED),
             (_cache(policy=m.POLICY_STATIC), 4, 4096, need, m.MOE_EUNSUPPORTED),
             (_cache(), 0, 4096, need, m.MOE_EINVAL),
             (_cache(), 4, None, need, m.MOE_EINVAL),
             (_cache(), 4, 4098, need, m.MOE_EINVAL),
             (_cache(), 4, 4096, need - 1, m.MOE_ECAPACITY),
             (_cache(slot_pool=4100), 4, 4096, need, m.MOE_EINVAL),
             (_cache(num_slots=0), 4, 4096, need, m.MOE_EINVAL)]
    for c, n, ws, wsb, code in cases:
        with pytest.raises(m.MoeError) as e:
            m.moe_cache_resize(sp, c, n, ws, wsb, stream=0)
        assert e.value.code == code
        assert c.num_slots in (0, 8)  # unchanged on failure


def test_ffn_argument_checks(L):
    s = _spec(has_shared=True)
    need = m.moe_ffn_workspace_bytes(s, 1)
    assert need > 0
    with pytest.raises(m.MoeError) as e:  # shared expert declared but not passed
        m.moe_expert_ffn(s, _cache(), 0, _plan(), 256, 1, 256, 256, None, 4096, need, 256,
                         stream=0)
    assert e.value.code == m.MOE_EINVAL
    with pytest.raises(m.MoeError) as e:  # workspace too small
        m.moe_expert_ffn(s, _cache(), 0, _plan(), 256, 1, 256, 256, 256, 4096, need - 1, 256,
                         stream=0)
    assert e.value.code == m.MOE_ECAPACITY
    with pytest.raises(m.MoeError) as e:  # workspace misaligned
        m.moe_expert_ffn(s, _cache(), 0, _plan(), 256, 1, 256, 256, 256, 4100, need, 256,
                         stream=0)
    assert e.value.code == m.MOE_EINVAL
    with pytest.raises(m.MoeError) as e:
        m.moe_expert_ffn(s, _cache(), 0, _plan(cap=200), 256, 65, 256, 256, 256, 4096, 1 << 30,
                         256, stream=0)
    assert e.value.code == m.MOE_EUNSUPPORTED


def test_layer_forward_argument_checks(L):
    s = _spec()
    need = m.moe_layer_workspace_bytes(s, 1)
    assert need >= m.moe_ffn_workspace_bytes(s, 1)
    with pytest.raises(m.MoeError) as e:
        m.moe_layer_forward(s, _cache(), 0, 256, 1, 256, None, None, _plan(), 256, 256, 4096,
                            need - 1, 256, stream=0)
    assert e.value.code == m.MOE_ECAPACITY
    with pytest.raises(m.MoeError) as e:
        m.moe_layer_forward(s, _cache(), 5, 256, 1, 256, None, None, _plan(), 256, 256, 4096,
                            need, 256, stream=0)
    assert e.value.code == m.MOE_EINVAL


def test_prefill_argument_checks(L):
    s = _spec(hidden=320 // 64 * 64)
    s.hidden = 320
    assert m.moe_prefill_workspace_bytes(s, 16) == 0  # hidden % 256 != 0
    s2 = _spec()
    assert m.moe_prefill_workspace_bytes(s2, 16) > 0
    with pytest.raises(m.MoeError) as e:
        m.moe_expert_ffn_prefill(s2, 4096, 4096, 16, 256, 256, None, None, 4096, 16, 4096,
                                 stream=0)
    assert e.value.code == m.MOE_ECAPACITY
    with pytest.raises(m.MoeError) as e:
        m.moe_expert_ffn_prefill(s2, None, 4096, 16, 256, 256, None, None, 4096, 1 << 30, 4096,
                                 stream=0)
    assert e.value.code == m.MOE_EINVAL
    for bank, layer, dst in ((4096, 7, 4096), (4096, -1, 4096), (None, 0, 4096), (4096, 0, None)):
        with pytest.raises(m.MoeError) as e:  # layer out of range, NULL bank or destination
            m.moe_layer_prefetch(s2, bank, layer, dst, stream=0)
        assert e.value.code == m.MOE_EINVAL
    assert m.moe_expert_ffn_prefill(s2, None, None, 0, None, None, None, None, None, 0, None,
                                    stream=0) == m.MOE_OK


def test_profile_argument_checks(L):
    s = _spec()
    need = m.moe_profile_workspace_bytes(s)
    assert need >= 2 * m.moe_expert_bytes(s)  # two blobs of copy scratch at least
    with pytest.raises(m.MoeError) as e:  # workspace too small
        m.moe_profile_bandwidths(s, _cache(), 0, 4096, need - 1, reps=2, stream=0)
    assert e.value.code == m.MOE_ECAPACITY
    with pytest.raises(m.MoeError) as e:  # layer out of range
        m.moe_profile_bandwidths(s, _cache(), 5, 4096, need, reps=2, stream=0)
    assert e.value.code == m.MOE_EINVAL
    with pytest.raises(m.MoeError) as e:
        m.moe_profile_bandwidths(s, _cache(), 0, 4096, need, reps=0, stream=0)
    assert e.value.code == m.MOE_EINVAL
    with pytest.raises(m.MoeError) as e:  # misaligned workspace
        m.moe_profile_bandwidths(s, _cache(), 0, 4100, need, reps=2, stream=0)
    assert e.value.code == m.MOE_EINVAL


def test_hot_placement_is_best_fixed_set():
    """hot_placement against brute force: on tiny traces no other set of S ids
    collects more static hits, and its order is count-descending, id-ascending."""
    import itertools

    import numpy as np

    from moe_expert_offload_gb300 import placement

    rng = np.random.default_rng(3)
    L, E, k = 2, 5, 2
    tr = np.stack([[rng.choice(E, size=k, replace=False) for _ in range(L)]
                   for _ in range(30)]).astype(np.int32)
    hits = lambda P: sum(int(l * E + e in P) for t in range(30) for l in range(L)
                         for e in set(tr[t, l].tolist()))
    for S in (1, 3, 6):
        got = placement.hot_placement(tr, E, S)
        best = max(hits(set(c)) for c in itertools.combinations(range(L * E), S))
        assert len(got) == S and hits(set(got.tolist())) == best
        cnt = [sum(int(u % E in tr[t, u // E]) for t in range(30)) for u in got]
        assert all((cnt[i], -got[i]) >= (cnt[i + 1], -got[i + 1]) for i in range(S - 1))
    assert list(placement.layer_placement(3, 4, 9)) == list(range(8))
    assert list(placement.layer_placement(3, 4, 100)) == list(range(12))
    assert placement.layer_placement(3, 4, 3).size == 0


def test_layer_kernel_count(L):
    """Host-side launch accounting of moe_layer_forward (no device work)."""
    c, cs = _cache(sync=None), _cache(sync=1 << 20)  # without / with sync words (K = 4)
    kc = m.moe_layer_kernel_count
    # sync words and T k <= 32, K <= 8, E <= 256: the whole step is one cooperative kernel
    assert kc(m.make_spec(1, 2048, 512, 256, 8), cs, 1) == 1
    assert kc(m.make_spec(1, 7168, 2048, 256, 8, router="sigmoid_group", n_groups=8,
                          topk_groups=4), cs, 4) == 1
    assert kc(m.make_spec(1, 2048, 512, 256, 8), cs, 8) == 3  # T k = 64 > 32
    assert kc(m.make_spec(1, 2048, 512, 256, 8), _cache(sync=1 << 20, k_victims=16), 1) == 3
    # logits, control step with the selection, one cooperative FFN kernel carrying the fill
    assert kc(m.make_spec(1, 2048, 512, 256, 8), c, 1) == 3
    assert kc(m.make_spec(1, 7168, 2048, 256, 8), c, 8) == 3
    # I % 512 != 0: the two streaming kernels (gate/up, down) carry the fill
    assert kc(m.make_spec(1, 2048, 256, 256, 8), cs, 1) == 4
    # H = 256 is below the streaming kernels' 512-column tiles: a fill copy kernel runs
    assert kc(m.make_spec(1, 256, 128, 16, 2), cs, 1) == 5
    assert kc(m.make_spec(1, 256, 128, 300, 2), cs, 1) == 6  # + select
    assert kc(m.make_spec(1, 2048, 512, 256, 8), cs, 9) == 5  # T > 8
    assert kc(m.make_spec(1, 2048, 512, 256, 8), cs, 0) == 0
    assert kc(m.make_spec(1, 2048, 512, 256, 8), cs, 65) == 0


def test_inject_hook_sets_and_clears(L):
    # host-side only: the flag is armed and cleared without any device work
    assert m.moe_debug_inject_ffn_stall(True) == m.MOE_OK
    assert m.moe_debug_inject_ffn_stall(False) == m.MOE_OK
