"""Pins for the oracle's number formats: bf16 rounding and the e4m3fn codec.

Independent references used here: torch's bfloat16 and float8_e4m3fn casts
(library routines), a brute-force nearest search over the 254 finite e4m3
codes, and closed forms that follow from the OCP E4M3 ("fn") definition:
bias 7, 3 mantissa bits, no infinities, largest finite 448, NaN at S.1111.111.
"""
import numpy as np
import pytest
import torch

import oracle

# ------------------------------------------------------------------ bf16


def _torch_bf16(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_round_matches_torch_random_bits():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2**32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    finite = np.isfinite(v)
    v = v[finite]
    np.testing.assert_array_equal(oracle.f32_to_bf16(v), _torch_bf16(v))


def test_bf16_round_ties_and_edges():
    # patterns whose low half is exactly 0x8000 (ties), just below and above
    hi = np.arange(0, 0x7f80, 7, dtype=np.uint32)
    lows = np.array([0x0000, 0x7fff, 0x8000, 0x8001, 0xffff], np.uint32)
    bits = ((hi[:, None] << 16) | lows[None, :]).ravel()
    bits = np.concatenate([bits, bits | 0x80000000])
    v = bits.view(np.float32)
    np.testing.assert_array_equal(oracle.f32_to_bf16(v), _torch_bf16(v))
    # ties go to the even upper half
    assert oracle.f32_to_bf16(np.array([1.0 + 2**-8], np.float32))[0] == 0x3F80
    assert oracle.f32_to_bf16(np.array([1.0 + 3 * 2**-8], np.float32))[0] == 0x3F82
    # overflow of the rounding carries to infinity
    assert oracle.f32_to_bf16(np.array([np.float32(3.4028235e38)], np.float32))[0] == 0x7F80


def test_bf16_to_f32_is_exact_widening():
    b = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = oracle.bf16_to_f32(b)
    same = (got.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(got) & np.isnan(ref))
    assert same.all()

# --------------------------------------------------------------- e4m3 fn


ALL_CODES = np.arange(256, dtype=np.uint32).astype(np.uint8)


def _torch_decode(c: np.ndarray) -> np.ndarray:
    return torch.from_numpy(c).view(torch.float8_e4m3fn).float().numpy()


def test_e4m3_decode_all_codes_match_torch():
    got = oracle.e4m3_decode(ALL_CODES)
    ref = _torch_decode(ALL_CODES)
    nan = np.isnan(ref)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.isnan(got[nan]).all()
    np.testing.assert_array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_roundtrip_all_finite_codes():
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    v = _torch_decode(finite)
    np.testing.assert_array_equal(oracle.e4m3_encode(v), finite)


def _brute_force_encode(v: np.ndarray) -> np.ndarray:
    """Nearest finite e4m3 code by exhaustive search; ties -> even code;
    magnitudes beyond 448 saturate; the sign is copied (also for zero)."""
    pos = np.arange(0, 0x7F, dtype=np.uint8)          # 0x00 .. 0x7E, ascending values
    pv = _torch_decode(pos).astype(np.float64)
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - pv[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among tied candidates prefer the even code (at most two tie)
    even = cand & ((pos[None, :] & 1) == 0)
    pick = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    code = pos[pick].astype(np.uint8)
    code[a > 448.0] = 0x7E
    return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)


def _boundary_values() -> np.ndarray:
    pos = _torch_decode(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float32)
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)  # exact in fp32
    vals = [pos, mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0)),
            np.nextafter(pos, np.float32(np.inf)), np.nextafter(pos, np.float32(0)),
            np.array([448.0, 456.0, 464.0, 470.0, 480.0, 1e6, 3e38, 2**-9, 2**-10, 3 * 2**-10,
                      2**-11, 2**-30, 1e-45], np.float32)]
    v = np.concatenate(vals).astype(np.float32)
    return np.concatenate([v, -v])


def test_e4m3_encode_boundaries_match_brute_force():
    v = _boundary_values()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), _brute_force_encode(v))


@pytest.mark.parametrize("seed", [0, 1])
def test_e4m3_encode_random_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = 500_000
    mag = np.exp2(rng.uniform(-12, 9.5, n)).astype(np.float32)
    v = np.where(rng.random(n) < 0.5, -mag, mag).astype(np.float32)
    got = oracle.e4m3_encode(v)
    for chunk in range(0, n, 50_000):
        sl = slice(chunk, chunk + 50_000)
        np.testing.assert_array_equal(got[sl], _brute_force_encode(v[sl]))


def test_e4m3_encode_matches_torch_within_range():
    # torch's cast rounds to nearest even; it is a library check for |v| <= 448
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(1_000_000) * 60).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), ref)


@pytest.mark.parametrize("v,code", [
    (448.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE), (-448.0, 0xFE),
    (2.0**-9, 0x01), (2.0**-10, 0x00), (3 * 2.0**-10, 0x02), (2.0**-6, 0x08),
    (1.0, 0x38), (1.0625, 0x38), (1.1875, 0x3A), (-0.0, 0x80), (0.0, 0x00),
    (240.0, 0x77), (float("nan"), 0x7F),
])
def test_e4m3_closed_forms(v, code):
    # 1.0 = 2^0 -> field 7, mantissa 0 -> 0x38; 1.0625 is the midpoint 1 .. 1.125 -> even 1.0;
    # 1.1875 is the midpoint 1.125 .. 1.25 -> even mantissa 2 (1.25) -> 0x3A;
    # 240 = 1.875 * 2^7 -> field 14, mantissa 7 -> 0x77.
    assert int(oracle.e4m3_encode(np.array([v], np.float32))[0]) == code
