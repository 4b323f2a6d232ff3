"""Shared helpers of the GPU parity tests (device marshalling, tolerances)."""
import numpy as np

# Expert-FFN tolerance: Edge0 §3.1 "math convention" compares every executor
# path elementwise with a dequantised reference at relative L2 < 1%; here also
# every element within 2% of the output's largest magnitude.
REL_L2 = 1e-2
ELEM = 2e-2


def assert_ffn_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / den if den > 0 else np.linalg.norm(got)
    worst = np.max(np.abs(got - ref)) if got.size else 0.0
    bound = ELEM * (np.max(np.abs(ref)) if ref.size else 0.0)
    assert rel <= REL_L2, f"{what}: relative L2 {rel:.3e} > {REL_L2}"
    assert worst <= bound, f"{what}: max |err| {worst:.3e} > {bound:.3e}"
    return rel


def dev_bits(t_bits, device):
    """uint16 bf16 bits (numpy) -> int16 device tensor with the same bytes."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(t_bits).view(np.int16)).to(device)


def dev(a, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def f32_bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
