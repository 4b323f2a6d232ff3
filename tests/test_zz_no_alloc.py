"""moe_expert_ffn_noalloc: the decode FFN for callers that cannot allocate
device memory (a host application that owns every device pool, a real-time
token loop that forbids allocation, a plugin handed only its input and output
buffers).  Its scratch is the library's built-in device array; this test calls
it through the C ABI and checks it against moe_expert_ffn (which takes a
caller workspace) on two consecutive decode steps, then checks that a size
needing more scratch than the array holds is refused."""
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

    _build.build()
    m.lib()


@pytest.mark.parametrize("H,I,E,T", [(2048, 512, 32, 1), (2048, 512, 32, 4),
                                     (2048, 512, 32, 16), (7168, 2048, 16, 8)])
def test_noalloc_matches_workspace_ffn_on_two_calls(H, I, E, T):
    """Qwen-shaped experts at 1, 4 and 16 tokens (16: past the cooperative
    kernel's 8, so the other FFN kernels run on the built-in array) and
    DeepSeek-shaped experts at 8 tokens."""
    k, S, K = 8, 12, 4
    spec = m.make_spec(1, H, I, E, k, has_shared=True)
    bank = synth.make_bank_torch(E + 1, H, I, 21, DEV)
    shared = bank[E]
    cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=bank[:E], device=DEV)
    plan = m.DevicePlan(T * k, K, device=DEV)
    wr = dev_bits(synth.router_weights(4, E, H), DEV)
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, k), dtype=torch.float32, device=DEV)
    wsb = m.moe_ffn_workspace_bytes(spec, T)
    assert wsb <= m.MOE_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    y_ws = torch.empty((T, H), dtype=torch.float32, device=DEV)
    y_na = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    xs = synth.ar1_stream(8, 2, H, n_streams=T)
    for step in range(2):
        x = dev_bits(xs[step], DEV)
        m.moe_route(spec, x, T, wr, None, logits, ids, wts)
        m.moe_cache_step(spec, cache.c, 0, ids, T, plan.c, 1)
        m.moe_expert_ffn(spec, cache.c, 0, plan.c, x, T, ids, wts, shared, ws, wsb, y_ws)
        m.moe_expert_ffn_noalloc(spec, cache.c, 0, plan.c, x, T, ids, wts, shared, y_na)
        torch.cuda.synchronize()
        assert_ffn_close(y_na.cpu().numpy(), y_ws.cpu().numpy(), f"call {step + 1}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    H, I, E, k, T = 7168, 2048, 256, 8, 64
    spec = m.make_spec(1, H, I, E, k)
    assert m.moe_ffn_workspace_bytes(spec, T) > m.MOE_NOALLOC_SCRATCH_BYTES
    bank = torch.empty(256, dtype=torch.uint8, device=DEV)
    cache = m.DeviceCache(spec, 1, 1, 1, 2, bank=bank, device=DEV, with_pool=False)
    cache.c.slot_pool = bank.data_ptr()
    plan = m.DevicePlan(T * k, 1, device=DEV)
    buf = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(m.MoeError) as e:
        m.moe_expert_ffn_noalloc(spec, cache.c, 0, plan.c, buf, T, buf, buf, None, buf)
    assert e.value.code == m.MOE_ECAPACITY
    assert "scratch" in str(e.value)
