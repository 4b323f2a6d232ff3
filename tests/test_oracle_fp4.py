"""Pins of the oracle's FP4 expert formats (MXFP4, NVFP4), the formats the
pages' deployed models use (FreeToken summary "Key results" table).  The FP8
E4M3 and E8M0 scale decoders are checked against torch's own conversions on
all 256 codes, the E2M1 elements against a hand-worked table, and the blob
dequantisation and expert math against closed forms and one-hot structures."""
import math
import os

import numpy as np
import pytest

from moe_expert_offload_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
torch = pytest.importorskip("torch")


def _same(a, b):
    return (math.isnan(a) and math.isnan(b)) or a == b


def test_e4m3_matches_torch(oracle):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    for b in range(256):
        assert _same(oracle.e4m3(b), ref[b]), b


def test_e8m0_matches_torch(oracle):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).tolist()
    for b in range(256):
        assert _same(oracle.e8m0(b), ref[b]), b


def test_e2m1_hand_worked_table(oracle):
    rows = [l.split("#")[0].split() for l in open(os.path.join(GOLD, "fp4_e2m1.txt"))]
    rows = [r for r in rows if r]
    assert len(rows) == 16
    for code, val in rows:
        got = oracle.e2m1(int(code))
        assert got == float(val) and math.copysign(1.0, got) == math.copysign(1.0, float(val))


def _blob_const(H, I, fmt, code, scale_byte, mat=(1.0, 1.0, 1.0)):
    B = synth.FP4_BLOCK[fmt]
    q = [np.full(shape, code, np.uint8) for shape in ((I, H), (I, H), (H, I))]
    s = [np.full((r, c // B), scale_byte, np.uint8) for r, c in ((I, H), (I, H), (H, I))]
    return synth.pack_fp4_blob(H, I, fmt, *q, *s, mat=mat)


def test_fp4_nibble_order(oracle):
    # byte 0x72: column 0 holds code 2 (1.0), column 1 code 7 (6.0); scale 1.0
    H, I = 64, 64
    blob = _blob_const(H, I, 0, 0, 127)
    blob[0] = 0x72
    w = oracle.fp4_blob_matrix(blob, H, I, 0, 0)
    assert w[0, 0] == 1.0 and w[0, 1] == 6.0 and np.all(w[0, 2:] == 0.0)


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp4_block_boundaries(oracle, fmt):
    # every block of a row gets its own scale: 2^j for block j (E8M0 127 + j, E4M3 exponent 7 + j)
    H, I = 128, 64
    B = synth.FP4_BLOCK[fmt]
    nb = H // B
    q = [np.full(shape, 2, np.uint8) for shape in ((I, H), (I, H), (H, I))]  # all 1.0
    blk = np.arange(nb)
    sg = np.tile((127 + blk) if fmt == 0 else ((7 + blk) << 3), (I, 1)).astype(np.uint8)
    s_other = [np.full((r, c // B), 127 if fmt == 0 else 0x38, np.uint8) for r, c in ((I, H), (H, I))]
    mat = (3.0, 1.0, 1.0)
    blob = synth.pack_fp4_blob(H, I, fmt, *q, sg, *s_other, mat=mat)
    w = oracle.fp4_blob_matrix(blob, H, I, 0, fmt)
    expect = np.repeat(2.0 ** blk, B) * (3.0 if fmt == 1 else 1.0)
    assert np.all(w == expect[None, :])
    assert np.all(oracle.fp4_blob_matrix(blob, H, I, 1, fmt) == 1.0)  # up: scale 1, mat 1


def test_fp4_formats_agree_on_power_of_two_scales(oracle):
    # an NVFP4 blob whose E4M3 block scales are powers of two and whose matrix scales
    # are 1 dequantises exactly like the MXFP4 blob with the same E8M0 exponents
    rng = np.random.default_rng(7)
    H, I = 128, 64
    q = [rng.integers(0, 16, size=s, dtype=np.uint8) for s in ((I, H), (I, H), (H, I))]
    ex = [rng.integers(-4, 5, size=(r, c // 32)) for r, c in ((I, H), (I, H), (H, I))]
    mx = [(127 + e).astype(np.uint8) for e in ex]
    nv = [np.repeat(((7 + e) << 3).astype(np.uint8), 2, axis=1) for e in ex]  # 2 x 16 = 32
    bm = synth.pack_fp4_blob(H, I, 0, *q, *mx)
    bn = synth.pack_fp4_blob(H, I, 1, *q, *nv, mat=(1.0, 1.0, 1.0))
    for which in range(3):
        assert np.array_equal(oracle.fp4_blob_matrix(bm, H, I, which, 0),
                              oracle.fp4_blob_matrix(bn, H, I, which, 1))


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp4_expert_closed_form(oracle, fmt):
    # all weights 1.0: g = u = sum(x), h = silu(g) * u for every row, y[o] = I * h
    H, I = 128, 64
    blob = _blob_const(H, I, fmt, 2, 127 if fmt == 0 else 0x38)
    x = synth.bf16_bits(np.random.default_rng(1).normal(0, 0.05, (2, H)))
    y = oracle.fp4_expert_forward(blob, H, I, fmt, x)
    for t in range(2):
        g = float(np.sum(synth.bf16_value(x[t]).astype(np.float64)))
        h = g / (1.0 + math.exp(-g)) * g
        assert np.allclose(y[t], I * h, rtol=1e-12, atol=0)


def test_fp4_expert_one_hot_structure(oracle):
    # gate[i0][c0] = 1, up[i0][c0] = 2, down[o0][i0] = 4, all else 0: only y[o0] is nonzero,
    # y[o0] = 4 * silu(x[c0]) * 2 x[c0]; a transposed or mis-indexed operand moves or loses it
    H, I, fmt = 128, 64, 1
    i0, c0, o0 = 5, 77, 100
    qg = np.zeros((I, H), np.uint8)
    qu = np.zeros((I, H), np.uint8)
    qd = np.zeros((H, I), np.uint8)
    qg[i0, c0], qu[i0, c0], qd[o0, i0] = 2, 4, 6
    s = [np.full((r, c // 16), 0x38, np.uint8) for r, c in ((I, H), (I, H), (H, I))]
    blob = synth.pack_fp4_blob(H, I, fmt, qg, qu, qd, *s)
    x = synth.bf16_bits(np.random.default_rng(2).normal(0, 1, (1, H)))
    y = oracle.fp4_expert_forward(blob, H, I, fmt, x)[0]
    xc = float(synth.bf16_value(x[0]).reshape(-1)[c0])
    expect = 4.0 * (xc / (1.0 + math.exp(-xc))) * 2.0 * xc
    assert y[o0] == pytest.approx(expect, rel=1e-14)
    assert np.count_nonzero(y) == (1 if expect != 0 else 0)


def test_fp4_rejects_bad_shapes(oracle):
    with pytest.raises(ValueError):
        oracle.fp4_blob_offsets(100, 64, 0)
    with pytest.raises(ValueError):
        oracle.fp4_blob_offsets(128, 64, 2)
