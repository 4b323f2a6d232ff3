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


@pytest.mark.parametrize("kw", [
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
    (dict(slot_pool=4100), m.MOE_EINVAL),
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
    with pytest.raises(m.MoeError) as e:
        m.moe_layer_prefetch(s2, 4096, 7, 4096, stream=0)
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
