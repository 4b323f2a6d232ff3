"""Seeded synthetic inputs for the MoE expert step.

This module only *generates data*: uniform int4 codes, bf16 scales and
biases, bf16 router weights, fp32 selection biases, AR(1) hidden-state
streams, prefill hidden states and Zipf routing traces, plus the byte packing
of one expert blob.  Nothing in it computes any part of the step (no routing,
no dequantisation, no matrix product), so the CPU oracle and the CUDA path can
both consume its output without sharing arithmetic.

All numpy generators are PCG64 (`numpy.random.default_rng(seed)`).  Floating
point values are rounded to bf16 with round-to-nearest-even before use.

Expert blob byte layout (one blob per (layer, expert), bank index l*E+e):
  Wg codes [I][H/2]  Wu codes [I][H/2]  Wd codes [H][I/2]      (uint8, 2 codes
  per byte, the low nibble holds the even column), then bf16 arrays
  Wg scales [I][H/64], Wg biases [I][H/64], Wu scales, Wu biases,
  Wd scales [H][I/64], Wd biases [H][I/64]; total rounded up to 256 bytes.
"""
from __future__ import annotations

import numpy as np

GROUP = 64
SECTION_ORDER = ("gq", "uq", "dq", "gs", "gb", "us", "ub", "ds", "db")


# ----------------------------------------------------------------- bf16 data
def bf16_bits(a) -> np.ndarray:
    """Round float values to bf16 (round-to-nearest-even); return uint16 bits."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    """uint16 bf16 bits -> float32 values (exact widening)."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------- blob packing
def blob_sections(H: int, I: int):
    """Byte offsets of the nine sections of one expert blob and its size."""
    if H % GROUP or I % GROUP:
        raise ValueError("hidden and intermediate sizes must be multiples of 64")
    sizes = {
        "gq": I * H // 2, "uq": I * H // 2, "dq": H * I // 2,
        "gs": I * (H // GROUP) * 2, "gb": I * (H // GROUP) * 2,
        "us": I * (H // GROUP) * 2, "ub": I * (H // GROUP) * 2,
        "ds": H * (I // GROUP) * 2, "db": H * (I // GROUP) * 2,
    }
    off, o = {}, 0
    for name in SECTION_ORDER:
        off[name] = o
        o += sizes[name]
    total = (o + 255) // 256 * 256
    return off, sizes, total


def pack_codes(q: np.ndarray) -> np.ndarray:
    """Pack int4 codes [rows][cols] (values 0..15) into bytes, low nibble = even col."""
    q = np.asarray(q, dtype=np.uint8)
    assert q.shape[-1] % 2 == 0 and q.max(initial=0) < 16
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def pack_blob(H, I, qg, qu, qd, sg, bg, su, bu, sd, bd) -> np.ndarray:
    """Assemble one expert blob from codes (0..15) and bf16 bit arrays."""
    off, sizes, total = blob_sections(H, I)
    blob = np.zeros(total, dtype=np.uint8)
    parts = {
        "gq": pack_codes(qg), "uq": pack_codes(qu), "dq": pack_codes(qd),
        "gs": np.asarray(sg, np.uint16), "gb": np.asarray(bg, np.uint16),
        "us": np.asarray(su, np.uint16), "ub": np.asarray(bu, np.uint16),
        "ds": np.asarray(sd, np.uint16), "db": np.asarray(bd, np.uint16),
    }
    for name in SECTION_ORDER:
        raw = np.ascontiguousarray(parts[name]).view(np.uint8).reshape(-1)
        assert raw.size == sizes[name], (name, raw.size, sizes[name])
        blob[off[name]:off[name] + raw.size] = raw
    return blob


def _scale_bias(rng, n):
    s = bf16_bits(rng.uniform(0.005, 0.02, size=n))
    b = bf16_bits(rng.uniform(-8.0, 8.0, size=n) * bf16_value(s))
    return s, b


def make_expert(rng, H: int, I: int) -> np.ndarray:
    """One random expert blob: codes U{0..15}, s~U[0.005,0.02], b=U[-8,8]*s."""
    qg = rng.integers(0, 16, size=(I, H), dtype=np.uint8)
    qu = rng.integers(0, 16, size=(I, H), dtype=np.uint8)
    qd = rng.integers(0, 16, size=(H, I), dtype=np.uint8)
    sg, bg = _scale_bias(rng, (I, H // GROUP))
    su, bu = _scale_bias(rng, (I, H // GROUP))
    sd, bd = _scale_bias(rng, (H, I // GROUP))
    return pack_blob(H, I, qg, qu, qd, sg, bg, su, bu, sd, bd)


def make_expert_bytes(rng, H: int, I: int) -> np.ndarray:
    """Same distribution as make_expert, drawn faster: code bytes are uniform
    (so both nibbles are uniform and independent)."""
    off, sizes, total = blob_sections(H, I)
    blob = np.zeros(total, dtype=np.uint8)
    blob[:off["gs"]] = rng.integers(0, 256, size=off["gs"], dtype=np.uint8)
    for sname, bname in (("gs", "gb"), ("us", "ub"), ("ds", "db")):
        n = sizes[sname] // 2
        s, b = _scale_bias(rng, n)
        blob[off[sname]:off[sname] + 2 * n] = s.view(np.uint8)
        blob[off[bname]:off[bname] + 2 * n] = b.view(np.uint8)
    return blob


def make_bank(n_experts: int, H: int, I: int, seed: int) -> np.ndarray:
    """Host bank of n_experts random blobs, uint8 [n_experts, S_e]."""
    rng = np.random.default_rng(seed)
    _, _, total = blob_sections(H, I)
    bank = np.empty((n_experts, total), dtype=np.uint8)
    for i in range(n_experts):
        bank[i] = make_expert(rng, H, I)
    return bank


def make_bank_torch(n_experts: int, H: int, I: int, seed: int, device):
    """Large bank generated directly in device memory with torch's RNG.

    Same distributions as make_bank; used where the bank is too large to build
    on the host (tens of GB).  Returns a uint8 tensor [n_experts, S_e].
    """
    import torch

    off, sizes, total = blob_sections(H, I)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    bank = torch.empty((n_experts, total), dtype=torch.uint8, device=device)
    chunk = max(1, min(n_experts, (1 << 30) // total))
    for a in range(0, n_experts, chunk):
        b = min(n_experts, a + chunk)
        blk = bank[a:b]
        blk[:, off["gq"]:off["gs"]].random_(0, 256, generator=g)
        end = off["db"] + sizes["db"]
        if total > end:
            blk[:, end:].zero_()
        for sname, bname in (("gs", "gb"), ("us", "ub"), ("ds", "db")):
            n = sizes[sname] // 2
            s = torch.rand((b - a, n), generator=g, device=device) * 0.015 + 0.005
            s = s.to(torch.bfloat16)
            bias = (torch.rand((b - a, n), generator=g, device=device) * 16.0 - 8.0) * s.float()
            blk[:, off[sname]:off[sname] + 2 * n].view(torch.bfloat16).copy_(s)
            blk[:, off[bname]:off[bname] + 2 * n].view(torch.bfloat16).copy_(bias.to(torch.bfloat16))
    return bank


# ---------------------------------------------------------- routing inputs
# ----------------------------------------------------------- FP4 experts
FP4_BLOCK = {0: 32, 1: 16}  # MXFP4: 32 elements per E8M0 scale; NVFP4: 16 per E4M3 scale


def fp4_blob_sections(H: int, I: int, fmt: int):
    """Byte offsets of an FP4 expert blob: codes Wg, Wu, Wd (as int4), one scale
    byte per block of each matrix, then (NVFP4) three fp32 matrix scales."""
    if H % GROUP or I % GROUP or fmt not in FP4_BLOCK:
        raise ValueError("hidden and intermediate sizes must be multiples of 64")
    B = FP4_BLOCK[fmt]
    sizes = {"gq": I * H // 2, "uq": I * H // 2, "dq": H * I // 2,
             "gs": I * H // B, "us": I * H // B, "ds": H * I // B, "mat": 12 if fmt == 1 else 0}
    off, o = {}, 0
    for name in ("gq", "uq", "dq", "gs", "us", "ds", "mat"):
        off[name] = o
        o += sizes[name]
    return off, sizes, (o + 255) // 256 * 256


def pack_fp4_blob(H, I, fmt, qg, qu, qd, sg, su, sd, mat=(1.0, 1.0, 1.0)) -> np.ndarray:
    """Assemble one FP4 expert blob from E2M1 codes (0..15) [rows][cols] and
    scale bytes [rows][cols / block] (E8M0 for MXFP4, E4M3 for NVFP4)."""
    off, sizes, total = fp4_blob_sections(H, I, fmt)
    blob = np.zeros(total, dtype=np.uint8)
    parts = {"gq": pack_codes(qg), "uq": pack_codes(qu), "dq": pack_codes(qd),
             "gs": np.asarray(sg, np.uint8), "us": np.asarray(su, np.uint8),
             "ds": np.asarray(sd, np.uint8)}
    if fmt == 1:
        parts["mat"] = np.asarray(mat, dtype="<f4").view(np.uint8)
    for name, arr in parts.items():
        flat = np.ascontiguousarray(arr).reshape(-1).view(np.uint8)
        assert flat.size == sizes[name], name
        blob[off[name]:off[name] + sizes[name]] = flat
    return blob


def make_fp4_expert(rng, H: int, I: int, fmt: int) -> np.ndarray:
    """Random FP4 expert: codes uniform over all 16, block scales around 2^-6
    (E8M0 bytes 118..124; E4M3 bytes with exponent field 1..5, no NaN), matrix
    scales U[0.5, 2) for NVFP4."""
    B = FP4_BLOCK[fmt]
    q = [rng.integers(0, 16, size=shape, dtype=np.uint8) for shape in ((I, H), (I, H), (H, I))]
    if fmt == 0:
        sc = [rng.integers(118, 125, size=(r, c // B), dtype=np.uint8)
              for r, c in ((I, H), (I, H), (H, I))]
    else:
        sc = [((rng.integers(1, 6, size=(r, c // B)) << 3) | rng.integers(0, 8, size=(r, c // B)))
              .astype(np.uint8) for r, c in ((I, H), (I, H), (H, I))]
    mat = tuple(float(v) for v in rng.uniform(0.5, 2.0, size=3)) if fmt == 1 else (1.0, 1.0, 1.0)
    return pack_fp4_blob(H, I, fmt, *q, *sc, mat=mat)


def make_fp4_bank_torch(n_experts: int, H: int, I: int, fmt: int, seed: int, device):
    """FP4 bank generated in device memory (torch's RNG), with the distributions of
    make_fp4_expert: codes uniform over all 16, E8M0 bytes 118..124 (MXFP4) or E4M3
    bytes with exponent field 1..5 (NVFP4), matrix scales U[0.5, 2) (NVFP4).
    fmt: 0 MXFP4, 1 NVFP4.  Returns a uint8 tensor [n_experts, S_e]."""
    import torch

    off, sizes, total = fp4_blob_sections(H, I, fmt)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    bank = torch.zeros((n_experts, total), dtype=torch.uint8, device=device)
    chunk = max(1, min(n_experts, (1 << 30) // total))
    for a in range(0, n_experts, chunk):
        b = min(n_experts, a + chunk)
        blk = bank[a:b]
        blk[:, off["gq"]:off["gs"]].random_(0, 256, generator=g)
        n_sc = off["mat"] - off["gs"]
        if fmt == 0:
            sc = torch.randint(118, 125, (b - a, n_sc), generator=g, device=device)
        else:
            e = torch.randint(1, 6, (b - a, n_sc), generator=g, device=device)
            m = torch.randint(0, 8, (b - a, n_sc), generator=g, device=device)
            sc = (e << 3) | m
        blk[:, off["gs"]:off["mat"]] = sc.to(torch.uint8)
        if fmt == 1:
            mat = torch.rand((b - a, 3), generator=g, device=device) * 1.5 + 0.5
            blk[:, off["mat"]:off["mat"] + 12].view(torch.float32).copy_(mat)
    return bank


def router_weights(seed: int, E: int, H: int, std: float = 0.02) -> np.ndarray:
    """bf16 bits [E][H], N(0, std)."""
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.normal(0.0, std, size=(E, H)))


def selection_bias(seed: int, E: int, std: float = 0.01) -> np.ndarray:
    """fp32 [E], N(0, std): added to sigmoid scores for expert selection only."""
    rng = np.random.default_rng(seed)
    return rng.normal(0.0, std, size=E).astype(np.float32)


def ar1_stream(seed: int, steps: int, H: int, n_streams: int = 1, rho: float = 0.9) -> np.ndarray:
    """AR(1) hidden states x_t = rho*x_{t-1} + eps_t, x_0 = eps_0, eps ~ N(0,1).

    The process runs in float64; each step is rounded to bf16.
    Returns uint16 bits [steps][n_streams][H].
    """
    rng = np.random.default_rng(seed)
    out = np.empty((steps, n_streams, H), dtype=np.uint16)
    x = np.zeros((n_streams, H))
    for t in range(steps):
        eps = rng.normal(0.0, 1.0, size=(n_streams, H))
        x = eps if t == 0 else rho * x + eps
        out[t] = bf16_bits(x)
    return out


def prefill_hidden(seed: int, T: int, H: int, w_router_bits: np.ndarray, boost: float = 3.0):
    """N(0,1) hidden states whose router logit for expert (t mod E) is raised by ~boost.

    Token t gets boost * W_r[e_t] / |W_r[e_t]|^2 added (e_t = t mod E), so the
    routing union of a long chunk covers every expert.  Returns bf16 bits [T][H].
    """
    rng = np.random.default_rng(seed)
    w = bf16_value(w_router_bits).astype(np.float64)
    E = w.shape[0]
    x = rng.normal(0.0, 1.0, size=(T, H))
    e = np.arange(T) % E
    x += boost * w[e] / np.sum(w[e] * w[e], axis=1, keepdims=True)
    return bf16_bits(x)


def zipf_trace(seed: int, steps: int, E: int, k: int, alpha: float = 1.1,
               overlap: float = 0.7, phase_steps: int | None = None) -> np.ndarray:
    """Synthetic routing trace int32 [steps][k] of distinct expert ids.

    Expert popularity is Zipf(alpha) over a random permutation of the experts.
    Step t keeps each of step t-1's experts with probability `overlap`, then
    tops up to k distinct experts with popularity-weighted draws without
    replacement.  With `phase_steps`, a new permutation is drawn every
    `phase_steps` steps (a change of task or workload phase: the popular
    experts change, the popularity curve does not).
    """
    rng = np.random.default_rng(seed)
    p_rank = 1.0 / np.arange(1, E + 1) ** alpha
    pop = np.empty(E)

    def draw_popularity():
        pop[rng.permutation(E)] = p_rank / p_rank.sum()

    draw_popularity()
    out = np.empty((steps, k), dtype=np.int32)
    prev: list[int] = []
    for t in range(steps):
        if phase_steps and t and t % phase_steps == 0:
            draw_popularity()
        keep = [e for e in prev if rng.random() < overlap]
        chosen = list(keep)
        avail = np.ones(E, dtype=bool)
        avail[chosen] = False
        while len(chosen) < k:
            p = np.where(avail, pop, 0.0)
            e = int(rng.choice(E, p=p / p.sum()))
            chosen.append(e)
            avail[e] = False
        out[t] = chosen
        prev = chosen
    return out
