"""Pins for the oracle's dispatch (bf16 and e4m3) and combine.

References independent of the oracle: round trips that must return the
input exactly (dispatch -> identity experts -> combine), the FP8 error
bound (at most half an e4m3 ulp of x/s, times s), closed forms (all-zero and
constant groups), hand-worked combine fixtures, and torch's float8_e4m3fn
decode (a library routine) for dequantisation.
"""
import json
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from combine_moedc_layout_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _decode(c):
    return torch.from_numpy(np.ascontiguousarray(c)).view(torch.float8_e4m3fn).float().numpy()


def _bf16(bits):
    return oracle.bf16_to_f32(bits)


def _run_layout(c):
    out = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    assert out["status"] == oracle.OK
    return out


# ------------------------------------------------------------- round trips

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_k1_unit_weight_roundtrip_is_exact(seed):
    c = synth.make_random_case(seed, T=40, H=256, K=1, E=7, R=7, cap=None, dtype=synth.BF16)
    lay = _run_layout(c)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=False)
    w = np.ones((c.T, 1), np.float32)
    y = oracle.combine(d["recv"], c.topk_idx, lay["slot"], w)["y"]
    np.testing.assert_array_equal(y, c.x)


@pytest.mark.parametrize("name", ["tiny", "imbalanced_small"])
def test_identity_experts_with_normalised_weights_return_x(name):
    if name == "tiny":
        c = synth.make_case("tiny")
    else:
        c = synth.make_case("imbalanced", T=256)
    lay = _run_layout(c)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=False)
    live = (c.topk_idx >= 0).astype(np.float32)
    w = c.topk_weights * live
    s = w.sum(axis=1, keepdims=True, dtype=np.float32)
    keep = s[:, 0] > 0
    w = np.where(s > 0, w / np.where(s > 0, s, 1), 0).astype(np.float32)
    y = oracle.combine(d["recv"], c.topk_idx, lay["slot"], w)["y"]
    # x is a bf16 value; sum_k w_k * x with sum_k w_k = 1 within a few binary32 ulps
    # lies far inside half a bf16 ulp of x, so rounding returns x exactly
    np.testing.assert_array_equal(y[keep], c.x[keep])
    assert (y[~keep] == 0).all()


def test_dispatch_bf16_rows_are_copies_of_source_tokens():
    c = synth.make_case("tiny")
    lay = _run_layout(c)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=False)
    for t in range(c.T):
        for k in range(c.K):
            e, s = c.topk_idx[t, k], lay["slot"][t, k]
            if e >= 0:
                np.testing.assert_array_equal(d["recv"][e, s], c.x[t])
                assert d["src_idx"][e, s] == t


# ------------------------------------------------------------------ FP8

def _e4m3_ulp(v):
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0**-6)))
    return np.where(a >= 2.0**-6, 2.0 ** (e - 3), 2.0**-9)


@pytest.mark.parametrize("name", ["low8", "default_ll"])
def test_fp8_dequant_error_bound(name):
    c = synth.make_case(name)
    lay = _run_layout(c)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    x = _bf16(c.x).astype(np.float64)
    G = c.G
    for t in range(c.T):
        for k in range(c.K):
            e, s = c.topk_idx[t, k], lay["slot"][t, k]
            q = _decode(d["recv"][e, s]).astype(np.float64).reshape(G, 128)
            sc = d["scales"][e, s].astype(np.float64)
            xr = x[t].reshape(G, 128)
            assert (sc > 0).all()
            # the scale maps the group's amax (clamped at 1e-4) near 448
            amax = np.maximum(np.abs(xr).max(axis=1), 1e-4)
            np.testing.assert_allclose(sc * 448.0, amax, rtol=2**-23)
            err = np.abs(xr - q * sc[:, None])
            bound = 0.5 * _e4m3_ulp(xr / sc[:, None]) * sc[:, None] * (1 + 2.0**-20)
            assert (err <= bound).all()


def test_fp8_zero_group_closed_form():
    T, H = 2, 256
    x = np.zeros((T, H), np.uint16)
    x[1, 128:] = synth.f32_to_bf16_bits(np.full(128, -3.0, np.float32))
    idx = np.array([[0], [1]], np.int32)
    lay = oracle.layout(idx, 2, 1, 1)
    d = oracle.dispatch(x, idx, lay["slot"], 2, 1, fp8=True)
    s0 = np.float32(1e-4) / np.float32(448.0)
    assert d["scales"][0, 0, 0] == s0 and d["scales"][0, 0, 1] == s0
    assert (d["recv"][0, 0] == 0).all()
    # token 1: group 0 is zero, group 1 is the constant -3 -> every code -448
    assert d["scales"][1, 0, 0] == s0
    assert d["scales"][1, 0, 1] == np.float32(3.0) / np.float32(448.0)
    assert (d["recv"][1, 0, 128:] == 0xFE).all()


@pytest.mark.parametrize("c_val", [1e-4, 0.37, 5.0, -7.25, 1000.0])
def test_fp8_constant_group_maps_to_max_code(c_val):
    x = synth.f32_to_bf16_bits(np.full((1, 128), c_val, np.float32))
    cb = _bf16(x)[0, 0]
    idx = np.array([[0]], np.int32)
    lay = oracle.layout(idx, 1, 1, 1)
    d = oracle.dispatch(x, idx, lay["slot"], 1, 1, fp8=True)
    code = 0x7E if cb > 0 else 0xFE
    if abs(cb) >= np.float32(1e-4):
        assert (d["recv"][0, 0] == code).all()
        assert d["scales"][0, 0, 0] == np.float32(abs(cb)) / np.float32(448.0)


def test_fp8_outlier_rows_do_not_touch_other_rows():
    c = synth.make_case("default_ll")
    rows = c.extra["outlier_rows"]
    assert len(rows) == 2
    lay = _run_layout(c)
    a = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    x2 = c.x.copy()
    x2[rows] = synth.f32_to_bf16_bits(_bf16(c.x[rows]) / np.float32(100.0))
    b = oracle.dispatch(x2, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    others = np.setdiff1d(np.arange(c.T), rows)
    for t in others[:40]:
        for k in range(c.K):
            e, s = c.topk_idx[t, k], lay["slot"][t, k]
            np.testing.assert_array_equal(a["recv"][e, s], b["recv"][e, s])
            np.testing.assert_array_equal(a["scales"][e, s], b["scales"][e, s])
    # the outlier rows carry ~100x larger scales
    e, s = c.topk_idx[rows[0], 0], lay["slot"][rows[0], 0]
    e2, s2 = c.topk_idx[rows[0], 0], lay["slot"][rows[0], 0]
    assert np.median(a["scales"][e, s] / b["scales"][e2, s2]) > 50


def test_fp8_unfilled_rows_untouched_and_src_idx_minus_one():
    c = synth.make_case("low4")
    lay = _run_layout(c)
    sentinel = np.full((c.E, c.cap, c.H), 0xAB, np.uint8)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True, recv=sentinel)
    cnt = lay["num_tokens_per_expert"]
    for e in range(c.E):
        assert (d["recv"][e, cnt[e]:] == 0xAB).all()
        assert (d["src_idx"][e, cnt[e]:] == -1).all()


# --------------------------------------------------------------- combine

def _hex_f32(h):
    return struct.unpack("<f", struct.pack("<I", int(h, 16)))[0]


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "combine_order.json")))["cases"],
                         ids=lambda c: c["name"])
def test_combine_golden(case):
    eo = np.array([int(h, 16) for h in case["expert_out_bf16_hex"]], np.uint16)
    eo = eo.reshape(case["E"], case["cap"], case["H"])
    w = np.array([_hex_f32(h) for h in case["weights_hex"]], np.float32).reshape(case["T"], case["K"])
    out = oracle.combine(eo, np.array(case["topk_idx"], np.int32), np.array(case["slot"], np.int32), w)
    np.testing.assert_array_equal(out["y"].reshape(-1), [int(h, 16) for h in case["y_bf16_hex"]])


def test_combine_all_masked_is_positive_zero():
    eo = np.full((2, 1, 64), 0x3F80, np.uint16)
    idx = np.full((3, 4), -1, np.int32)
    y = oracle.combine(eo, idx, idx.copy(), np.ones((3, 4), np.float32))["y"]
    assert (y == 0).all()


def test_combine_k1_is_scaled_gather():
    c = synth.make_random_case(5, T=30, H=128, K=1, E=4, R=2, cap=None, dtype=synth.BF16)
    lay = _run_layout(c)
    eo = synth.make_expert_out(c, 5)
    w = np.full((c.T, 1), 2.0, np.float32)  # a power of two: the product is exact
    y = oracle.combine(eo, c.topk_idx, lay["slot"], w)["y"]
    for t in range(c.T):
        e, s = c.topk_idx[t, 0], lay["slot"][t, 0]
        ref = synth.f32_to_bf16_bits(_bf16(eo[e, s]) * np.float32(2.0))
        np.testing.assert_array_equal(y[t], ref)


def test_combine_close_to_float64_sum():
    c = synth.make_case("tiny")
    lay = _run_layout(c)
    eo = synth.make_expert_out(c, 0)
    y = _bf16(oracle.combine(eo, c.topk_idx, lay["slot"], c.topk_weights)["y"]).astype(np.float64)
    ref = np.zeros((c.T, c.H))
    for t in range(c.T):
        for k in range(c.K):
            e = c.topk_idx[t, k]
            if e >= 0:
                ref[t] += float(c.topk_weights[t, k]) * _bf16(eo[e, lay["slot"][t, k]]).astype(np.float64)
    # bf16 rounding (2^-9 relative) dominates the K binary32 roundings
    tol = np.abs(ref) * (2.0**-8) + 1e-30
    assert (np.abs(y - ref) <= tol).all()


def test_combine_skips_slots_beyond_capacity():
    eo = np.full((1, 1, 8), 0x3F80, np.uint16)          # 1.0 everywhere
    idx = np.array([[0, 0]], np.int32)
    slot = np.array([[0, 1]], np.int32)                  # slot 1 >= cap = 1: dropped
    y = oracle.combine(eo, idx, slot, np.array([[1.0, 1.0]], np.float32))["y"]
    assert (y == 0x3F80).all()


def test_fp8_quotient_is_one_rounded_division():
    """Pins the reading 'v = x / s' (one binary32 division per element)
    against the plausible 'v = x * (1 / s)': pick groups where the two give
    different e4m3 codes and check the oracle sides with the division, whose
    code is found by exhaustive nearest search."""
    rng = np.random.default_rng(11)
    found = 0
    for _ in range(200):
        g = synth.f32_to_bf16_bits(rng.standard_normal(128).astype(np.float32))
        xf = _bf16(g)
        amax = np.float32(max(np.abs(xf).max(), np.float32(1e-4)))
        s = np.float32(amax / np.float32(448.0))
        div = (xf / s).astype(np.float32)
        mul = (xf * np.float32(np.float32(1.0) / s)).astype(np.float32)
        from test_oracle_codec import _brute_force_encode
        cd, cm = _brute_force_encode(div), _brute_force_encode(mul)
        if (cd != cm).any():
            idx = np.array([[0]], np.int32)
            d = oracle.dispatch(g.reshape(1, 128), idx, np.array([[0]], np.int32), 1, 1, fp8=True)
            np.testing.assert_array_equal(d["recv"][0, 0], cd)
            assert (d["recv"][0, 0] != cm).any()
            found += 1
    assert found >= 3


# --------------------------------------------------------------- dequant

@pytest.mark.parametrize("code,scale,expect", [
    (0x7E, 2.0, 896.0), (0xFE, 0.25, -112.0), (0x01, 1.0, 2.0**-9), (0x00, 3.0, 0.0),
    (0x38, 1.5, 1.5), (0x3A, 0.5, 0.625),
])
def test_dequant_closed_forms(code, scale, expect):
    r = np.full((1, 1, 128), code, np.uint8)
    out = oracle.dequant_e4m3(r, np.array([[[scale]]], np.float32), np.array([1], np.int32))
    assert _bf16(out[0, 0, :1])[0] == np.float32(expect)


def test_dequant_matches_torch_decode_multiply_cast():
    rng = np.random.default_rng(21)
    E, cap, H = 3, 5, 256
    codes = rng.integers(0, 256, (E, cap, H), dtype=np.int64).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11                 # dispatch never writes NaN codes
    sc = np.exp(rng.uniform(-20, 5, (E, cap, H // 128))).astype(np.float32)
    cnt = np.array([5, 2, 0], np.int32)
    got = oracle.dequant_e4m3(codes, sc, cnt)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).float()
    ref = (dec * torch.from_numpy(np.repeat(sc, 128, axis=2))).to(torch.bfloat16)
    ref = ref.view(torch.int16).numpy().view(np.uint16)
    for e in range(E):
        np.testing.assert_array_equal(got[e, :cnt[e]], ref[e, :cnt[e]])
        assert (got[e, cnt[e]:] == 0).all()                # rows past the count untouched


def test_dispatch_then_dequant_error_bound():
    c = synth.make_case("low8")
    lay = _run_layout(c)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    deq = oracle.dequant_e4m3(d["recv"], d["scales"], lay["num_tokens_per_expert"])
    x = _bf16(c.x).astype(np.float64)
    for t in range(c.T):
        for k in range(c.K):
            e, s = c.topk_idx[t, k], lay["slot"][t, k]
            y = _bf16(deq[e, s]).astype(np.float64)
            sc = np.repeat(d["scales"][e, s].astype(np.float64), 128)
            # e4m3 half-ulp of x/s times s, plus the bf16 rounding of the product
            bound = 0.5 * _e4m3_ulp(x[t] / sc) * sc * (1 + 2.0**-20) + np.abs(y) * 2.0**-8
            assert (np.abs(y - x[t]) <= bound).all()


# ------------------------------------------------------------ e4m3 combine

def test_combine_e4m3_k1_unit_weight_equals_dequant():
    """One entry with weight 1: the sum is the dequantised value itself."""
    c = synth.make_random_case(71, T=60, H=256, K=1, E=6, R=3, cap=None, dtype=synth.FP8_E4M3)
    lay = _run_layout(c)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    w = np.ones((c.T, 1), np.float32)
    y = oracle.combine_e4m3(d["recv"], d["scales"], c.topk_idx, lay["slot"], w)["y"]
    deq = oracle.dequant_e4m3(d["recv"], d["scales"], lay["num_tokens_per_expert"])
    for t in range(c.T):
        np.testing.assert_array_equal(y[t], deq[c.topk_idx[t, 0], lay["slot"][t, 0]])


def test_combine_e4m3_column_major_scales_same_result():
    c = synth.make_case("low8")
    lay = _run_layout(c)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    a = oracle.combine_e4m3(d["recv"], d["scales"], c.topk_idx, lay["slot"], c.topk_weights)
    cm = np.ascontiguousarray(d["scales"].transpose(0, 2, 1))           # [E, G, cap]
    b = oracle.combine_e4m3(d["recv"], cm, c.topk_idx, lay["slot"], c.topk_weights,
                            scale_cols=True)
    np.testing.assert_array_equal(a["y"], b["y"])


def test_combine_e4m3_identity_round_trip_near_x():
    """Identity experts (expert output = the dispatched e4m3 rows) and weights
    renormalised to sum 1 return x within the e4m3 error of each group."""
    c = synth.make_case("low16")
    w = c.topk_weights / c.topk_weights.sum(axis=1, keepdims=True, dtype=np.float32)
    lay = _run_layout(c)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    y = oracle.combine_e4m3(d["recv"], d["scales"], c.topk_idx, lay["slot"],
                            w.astype(np.float32))["y"]
    x = _bf16(c.x).astype(np.float64)
    yy = _bf16(y).astype(np.float64)
    amax = np.abs(x).reshape(c.T, -1, 128).max(axis=2).repeat(128, axis=1)
    assert (np.abs(yy - x) <= amax * 2.0**-4 + np.abs(x) * 2.0**-7).all()


def test_combine_e4m3_closed_form():
    # codes 0x7E (448) and 0x38 (1.0) with scales 0.5 and 4; weights 0.25, 0.5
    q = np.array([[[0x7E] * 128], [[0x38] * 128]], np.uint8)                # [E=2, cap=1, H=128]
    s = np.array([[[0.5]], [[4.0]]], np.float32)
    idx = np.array([[0, 1]], np.int32)
    slot = np.array([[0, 0]], np.int32)
    w = np.array([[0.25, 0.5]], np.float32)
    y = oracle.combine_e4m3(q, s, idx, slot, w)["y"]
    # 0.25 * 224 + 0.5 * 4 = 58 exactly
    assert (_bf16(y) == np.float32(58.0)).all()
