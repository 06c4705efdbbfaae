"""Pins for the oracle's per-token e4m3 variants: dispatch with one scale
per token row, its dequantisation, and combine from e4m3 rows with per-row
scales.

References independent of the per-token code: the per-128 dispatch at
H = 128 (where the two rules coincide), the monotonicity of a correctly
rounded division (the row scale is the largest of the row's group scales),
closed forms (the row maximum lands on +-448; an all-zero row), the e4m3
error bound, and torch's float8_e4m3fn / bfloat16 casts (library routines).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moedc_layout_gb300 import synth


def _bf16(bits):
    return oracle.bf16_to_f32(bits)


def _decode(c):
    return torch.from_numpy(np.ascontiguousarray(c)).view(torch.float8_e4m3fn).float().numpy()


def _e4m3_ulp(v):
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0**-6)))
    return np.where(a >= 2.0**-6, 2.0 ** (e - 3), 2.0**-9)


def _chain(c):
    lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    assert lay["status"] == oracle.OK
    d = oracle.dispatch_token_scale(c.x, c.topk_idx, lay["slot"], c.E, c.cap)
    assert d["status"] == oracle.OK
    return lay, d


def _filled(c, lay):
    """(t, e, s) of every entry that received a row."""
    out = []
    for t in range(c.T):
        for k in range(c.K):
            e, s = int(c.topk_idx[t, k]), int(lay["slot"][t, k])
            if 0 <= e < c.E and 0 <= s < c.cap:
                out.append((t, e, s))
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_h128_equals_per_group_dispatch(seed):
    c = synth.make_random_case(30 + seed, T=90, H=128, K=4, E=12, R=4, cap=None,
                               dtype=synth.FP8_E4M3, mask_p=0.1)
    lay, d = _chain(c)
    g = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    np.testing.assert_array_equal(d["recv"], g["recv"])
    np.testing.assert_array_equal(d["src_idx"], g["src_idx"])
    np.testing.assert_array_equal(d["scales"].view(np.uint32), g["scales"][:, :, 0].view(np.uint32))


@pytest.mark.parametrize("name", ["low8", "default_ll"])
def test_row_scale_is_largest_group_scale(name):
    """RN(max(a, 1e-4) / 448) is monotone in a, so the row scale is exactly
    the largest of the per-128 scales of the same row."""
    c = synth.make_case(name)
    lay, d = _chain(c)
    g = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    for t, e, s in _filled(c, lay):
        assert d["scales"][e, s] == g["scales"][e, s].max()


@pytest.mark.parametrize("name", ["low8", "default_ll"])
def test_row_maximum_encodes_to_448(name):
    c = synth.make_case(name)
    lay, d = _chain(c)
    x = _bf16(c.x)
    for t, e, s in _filled(c, lay):
        a = np.abs(x[t])
        at = np.nonzero(a == a.max())[0]
        want = np.where(x[t, at] < 0, 0xFE, 0x7E)
        np.testing.assert_array_equal(d["recv"][e, s, at], want)


def test_zero_row_closed_form():
    x = np.zeros((2, 384), np.uint16)
    x[1] = synth.f32_to_bf16_bits(np.linspace(-2.0, 1.0, 384, dtype=np.float32))
    idx = np.array([[0], [1]], np.int32)
    slot = np.array([[0], [0]], np.int32)
    d = oracle.dispatch_token_scale(x, idx, slot, 2, 1)
    assert d["scales"][0, 0] == np.float32(np.float32(1e-4) / np.float32(448.0))
    assert (d["recv"][0, 0] == 0).all()
    assert d["scales"][1, 0] == np.float32(np.float32(2.0) / np.float32(448.0))
    assert d["recv"][1, 0, 0] == 0xFE


@pytest.mark.parametrize("name", ["low16", "default_ll"])
def test_error_bound_and_torch_cast(name):
    """Every code is torch's e4m3fn cast of the binary32 quotient x / s, and
    |x - q s| is at most half an e4m3 ulp of x / s, times s."""
    c = synth.make_case(name)
    lay, d = _chain(c)
    x32 = _bf16(c.x)
    for t, e, s in _filled(c, lay):
        sc = d["scales"][e, s]
        v = (x32[t] / sc).astype(np.float32)
        ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(d["recv"][e, s], ref)
        q = _decode(d["recv"][e, s]).astype(np.float64)
        err = np.abs(x32[t].astype(np.float64) - q * float(sc))
        assert (err <= 0.5 * _e4m3_ulp(v) * float(sc) * (1 + 2.0**-20)).all()


def test_unfilled_rows_untouched_and_src_idx():
    c = synth.make_random_case(33, T=40, H=256, K=3, E=9, R=3, cap=None, dtype=synth.FP8_E4M3,
                               mask_p=0.2)
    lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    init = np.full((c.E, c.cap, c.H), 0xA5, np.uint8)
    d = oracle.dispatch_token_scale(c.x, c.topk_idx, lay["slot"], c.E, c.cap, recv=init.copy())
    g = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    np.testing.assert_array_equal(d["src_idx"], g["src_idx"])
    filled = d["src_idx"] >= 0
    assert (d["recv"][~filled] == 0xA5).all()


def test_dequant_token_matches_torch_decode_multiply_cast():
    c = synth.make_case("low16")
    lay, d = _chain(c)
    cnt = lay["num_tokens_per_expert"]
    out = oracle.dequant_e4m3_token(d["recv"], d["scales"], cnt)
    dec = torch.from_numpy(d["recv"]).view(torch.float8_e4m3fn).float()
    ref = (dec * torch.from_numpy(d["scales"])[:, :, None]).to(torch.bfloat16)
    ref = ref.view(torch.int16).numpy().view(np.uint16)
    for e in range(c.E):
        n = min(int(cnt[e]), c.cap)
        np.testing.assert_array_equal(out[e, :n], ref[e, :n])
        assert (out[e, n:] == 0).all()


def test_combine_e4m3_per_token_equals_broadcast_group_scales():
    c = synth.make_case("low8")
    lay, d = _chain(c)
    a = oracle.combine_e4m3(d["recv"], d["scales"], c.topk_idx, lay["slot"], c.topk_weights,
                            per_token=True)
    wide = np.ascontiguousarray(np.repeat(d["scales"][:, :, None], c.G, axis=2))
    b = oracle.combine_e4m3(d["recv"], wide, c.topk_idx, lay["slot"], c.topk_weights)
    assert a["status"] == b["status"] == oracle.OK
    np.testing.assert_array_equal(a["y"], b["y"])


def test_combine_e4m3_per_token_k1_unit_weight_equals_dequant():
    c = synth.make_random_case(34, T=50, H=384, K=1, E=5, R=5, cap=None, dtype=synth.FP8_E4M3)
    lay, d = _chain(c)
    y = oracle.combine_e4m3(d["recv"], d["scales"], c.topk_idx, lay["slot"],
                            np.ones((c.T, 1), np.float32), per_token=True)["y"]
    deq = oracle.dequant_e4m3_token(d["recv"], d["scales"], lay["num_tokens_per_expert"])
    for t in range(c.T):
        np.testing.assert_array_equal(y[t], deq[c.topk_idx[t, 0], lay["slot"][t, 0]])


def test_hand_worked_row():
    """One row whose maximum is 7, so s = 7 / 448 = 2^-6 exactly and every
    quotient x / s is exact; the codes follow from the e4m3fn grid by hand:
    448 -> 0x7E; -224 = -1.75 * 2^7 -> 0xF6; 112 = 1.75 * 2^6 -> 0x6E;
    28 = 1.75 * 2^4 -> 0x5E; bf16(0.1) / s = 6.40625 lies between 6.0 and 6.5
    (spacing 0.5 in [4, 8)) and rounds to 6.5 = 1.625 * 2^2 -> 0x4D;
    bf16(1e-4) / s = 0.0064087 is 3.28 subnormal steps of 2^-9 -> 0x03; 0 -> 0x00."""
    vals = np.zeros(128, np.float32)
    vals[:7] = [7.0, -3.5, 1.75, 0.4375, 0.1, 1e-4, 0.0]
    x = synth.f32_to_bf16_bits(vals).reshape(1, 128)
    d = oracle.dispatch_token_scale(x, np.array([[0]], np.int32), np.array([[0]], np.int32), 1, 1)
    assert d["scales"][0, 0] == np.float32(2.0**-6)
    assert [int(v) for v in d["recv"][0, 0, :7]] == [0x7E, 0xF6, 0x6E, 0x5E, 0x4D, 0x03, 0x00]
    assert (d["recv"][0, 0, 7:] == 0).all()
