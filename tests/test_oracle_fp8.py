"""Pins of the FP8 E4M3 oracle against things other than itself: PyTorch's float8_e4m3fn
type (an independent implementation of the same format) for every code's value and for the
rounding of in-range values including every tie, the format's printed constants, and a
brute-force matmul over decoded codes."""
import numpy as np
import pytest

from oracle import fp8 as F

torch = pytest.importorskip("torch")
if not hasattr(torch, "float8_e4m3fn"):
    pytest.skip("torch without float8_e4m3fn", allow_module_level=True)


def torch_codes(v):
    return torch.tensor(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_every_code_matches_torch():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(F.DECODE))
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ref[~nan], F.DECODE[~nan])


def test_encode_matches_torch_in_range_and_on_ties():
    """Random values in (−448, 448), every code's value and every midpoint between adjacent
    codes (the ties, where round-to-nearest-even decides)."""
    rng = np.random.default_rng(0)
    vals = [rng.uniform(-448, 448, 4000), rng.normal(size=4000) * 2.0 ** rng.integers(-12, 8, 4000)]
    pos = F.DECODE[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    vals += [pos, -pos, mids, -mids]
    v = np.concatenate(vals).astype(np.float32)
    v = v[np.abs(v) <= 448]
    assert np.array_equal(F.encode(v), torch_codes(v))


def test_printed_constants_and_saturation():
    """1 → 0x38, 448 → 0x7E (the largest finite), 2⁻⁹ → 0x01 (the smallest subnormal), ±0;
    ties: 2⁻¹⁰ → 0x00 and 3·2⁻¹⁰ → 0x02 (even codes); beyond ±448 saturates; NaN → 0x7F."""
    cases = [(1.0, 0x38), (448.0, 0x7E), (2.0 ** -9, 0x01), (0.0, 0x00), (-0.0, 0x80), (2.0 ** -10, 0x00),
             (3 * 2.0 ** -10, 0x02), (460.0, 0x7E), (1e9, 0x7E), (-1e9, 0xFE), (2.0 ** -6, 0x08), (240.0, 0x77)]
    for v, c in cases:
        assert int(F.encode([v])[0]) == c, (v, hex(int(F.encode([v])[0])))
    assert int(F.encode([np.nan])[0]) == 0x7F


def test_quantize_amax_maps_to_max():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(33, 17)).astype(np.float32) * 3
    codes, scale = F.quantize(x)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert F.decode(codes)[i] == np.sign(x[i]) * 448.0
    back = F.decode(codes) / scale
    normal = np.abs(x) * scale >= 2.0 ** -6
    assert np.all(np.abs(back - x)[normal] <= np.abs(x)[normal] * 2.0 ** -4)
    assert F.quantize(np.zeros(5))[1] == 1.0


def test_matmul_brute_force():
    rng = np.random.default_rng(2)
    A = rng.integers(0, 256, (5, 7)).astype(np.uint8)
    B = rng.integers(0, 256, (3, 7)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x38
    B[(B & 0x7F) == 0x7F] = 0x38
    C = F.matmul_fp8(A, B, alpha=0.5, inv_scale_a=0.25, inv_scale_b=2.0)
    for i in range(5):
        for j in range(3):
            s = sum(F.decode_code(int(A[i, k])) * 0.25 * F.decode_code(int(B[j, k])) * 2.0 for k in range(7))
            assert C[i, j] == pytest.approx(0.5 * s, rel=1e-15, abs=1e-300)
