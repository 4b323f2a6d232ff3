"""The checked build (libmoe_checked.so, -DMOE_CHECKED): device-side range
checks on the cache-table entries the kernels read.  Run in a child process that
loads the checked library (MOE_LIBRARY).  With intact tables the checked build
gives the oracle's routing, plans and outputs with no error bit; with an entry
of slot_of_id corrupted to a value past the pool, the step ORs MOE_DERR_RANGE
into plan.err, treats the entry as absent (the expert is a miss) and finishes;
after a cache reset the next steps are normal again."""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r'''
import sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
sys.path.insert(0, HERE)
import moe_expert_offload_gb300 as m
from moe_expert_offload_gb300 import synth
import oracle
from gpu_util import assert_ffn_close, dev, dev_bits

oracle.build()
DEV = "cuda:0"
assert m.library_path().endswith("libmoe_checked.so")
for sync in (True, False):
    H, I, E, k, T, S, K = 1024, 512, 16, 4, 1, 6, 3
    spec = m.make_spec(1, H, I, E, k, has_shared=True)
    bank_h = synth.make_bank(E + 1, H, I, 5)
    bank = dev(bank_h, DEV)
    cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=bank[:E], device=DEV, sync=sync)
    plan = m.DevicePlan(T * k, K, device=DEV)
    wsb = m.moe_layer_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    y = torch.empty((T, H), dtype=torch.float32, device=DEV)
    wr_h = synth.router_weights(3, E, H)
    wr = dev_bits(wr_h, DEV)
    ost = oracle.CacheState(E, S)
    rng = np.random.default_rng(2)
    for step in range(8):
        xb = synth.bf16_bits(rng.normal(0, 1.5, (T, H)))
        oid, ow = oracle.route_softmax_topk(oracle.router_logits(xb, wr_h), k)
        corrupt = step == 5
        if corrupt:  # a routed expert's table entry now points past the pool
            cache.slot_of_id[int(oid[0, 0])] = 1 << 30
        m.moe_layer_forward(spec, cache.c, 0, dev_bits(xb, DEV), T, wr, None, bank[E], plan.c,
                            ids, wts, ws, wsb, y)
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), oid)
        err = int(plan.err[0].item())
        ref = oracle.moe_ffn(list(bank_h[:E]), H, I, xb, oid, ow, bank_h[E], I)
        if corrupt:
            assert err & m.MOE_DERR_RANGE, err
            assert np.all(np.isfinite(y.cpu().numpy()))
            assert_ffn_close(y.cpu().numpy(), ref, "corrupted entry read from the bank")
            plan.err.zero_()
            m.moe_cache_reset(spec, cache.c)
            ost = oracle.CacheState(E, S)
            continue
        assert err == 0, err
        op = oracle.cache_step(ost, E, 0, oid, K, 52700, 77300)
        assert int(plan.counts[4].item()) == op["n_fill"]
        assert_ffn_close(y.cpu().numpy(), ref, f"step {step}")
print("checked build ok")
'''


def test_checked_build_flags_bad_table_entries_and_matches_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_offload_gb300 import _build
    import oracle

    oracle.build()
    lib = _build.build(checked=True)
    env = dict(os.environ, MOE_LIBRARY=lib)
    code = f"ROOT = {ROOT!r}\nHERE = {HERE!r}\n" + CHILD
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=900)
    assert p.returncode == 0, (p.stdout + p.stderr)[-4000:]
    assert "checked build ok" in p.stdout
