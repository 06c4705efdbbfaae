"""Helpers for GPU-vs-oracle parity tests: move seeded inputs to the device,
run the library through its C ABI, run the oracle on the same bytes and
compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_moedc_layout_gb300 import moedc, synth


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bits_host(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a device tensor (bf16 -> uint16, e4m3 -> uint8)."""
    t = t.detach().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).cpu().numpy()
    return t.cpu().numpy()


class DevCase:
    """A synth.Case resident on the GPU."""

    def __init__(self, c: synth.Case):
        self.c = c
        self.x = bf16_dev(c.x) if c.T > 0 else torch.empty((0, c.H), dtype=torch.bfloat16,
                                                             device="cuda")
        self.topk_idx = torch.from_numpy(c.topk_idx).cuda()
        self.topk_weights = torch.from_numpy(c.topk_weights).cuda()


def run_layout(d: DevCase, status: torch.Tensor | None = None) -> moedc.Layout:
    c = d.c
    return moedc.layout(d.topk_idx, c.E, c.R, c.cap, status=status)


def compare_layout(lay: moedc.Layout, ref: dict, T: int) -> None:
    np.testing.assert_array_equal(lay.num_tokens_per_expert.cpu().numpy(),
                                  ref["num_tokens_per_expert"])
    np.testing.assert_array_equal(lay.num_tokens_per_rank.cpu().numpy(), ref["num_tokens_per_rank"])
    if T > 0:
        np.testing.assert_array_equal(lay.is_token_in_rank.cpu().numpy(), ref["is_token_in_rank"])
        np.testing.assert_array_equal(lay.slot.cpu().numpy(), ref["slot"])
    assert int(lay.status.item()) == ref["status"]


def valid_rows(cnt: np.ndarray, cap: int) -> np.ndarray:
    """Flat row indices e*cap + s of [E, cap] rows that some entry fills."""
    E = cnt.shape[0]
    fill = np.minimum(cnt, cap)
    return np.concatenate([e * cap + np.arange(fill[e]) for e in range(E)]).astype(np.int64) \
        if fill.sum() else np.zeros(0, np.int64)


def compare_dispatch(c: synth.Case, recv: torch.Tensor, scales, src_idx: torch.Tensor,
                     ref_lay: dict, ref: dict) -> None:
    np.testing.assert_array_equal(src_idx.cpu().numpy(), ref["src_idx"])
    rows = valid_rows(ref_lay["num_tokens_per_expert"], c.cap)
    if rows.size == 0:
        return
    ridx = torch.from_numpy(rows).cuda()
    got = bits_host(recv.reshape(c.E * c.cap, c.H).index_select(0, ridx))
    want = ref["recv"].reshape(c.E * c.cap, c.H)[rows]
    np.testing.assert_array_equal(got, want)
    if c.dtype == synth.FP8_E4M3:
        gs = scales.reshape(c.E * c.cap, c.G).index_select(0, ridx).cpu().numpy()
        ws = ref["scales"].reshape(c.E * c.cap, c.G)[rows]
        np.testing.assert_array_equal(gs.view(np.uint32), ws.view(np.uint32))


def bf16_ulp(ref_bits: np.ndarray) -> np.ndarray:
    """One bf16 ulp at each reference value: 2^(floor(log2|y|) - 7) for normal
    values, the subnormal spacing 2^-133 below the smallest normal."""
    v = oracle.bf16_to_f32(ref_bits).astype(np.float64)
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0**-126, 2.0 ** (e - 7), 2.0**-133)


def compare_combine(y: torch.Tensor, ref_y: np.ndarray) -> None:
    """The gate: |y - y_ref| <= 1 bf16 ulp of |y_ref| (zero must match as +-0).
    The kernel follows the oracle's exact operation order, so it is also
    expected to be bit-exact; that is asserted separately."""
    got = bits_host(y)
    g = oracle.bf16_to_f32(got).astype(np.float64)
    r = oracle.bf16_to_f32(ref_y).astype(np.float64)
    ulp = bf16_ulp(ref_y)
    zero = r == 0
    assert (g[zero] == 0).all()
    assert (np.abs(g - r)[~zero] <= ulp[~zero]).all()
    np.testing.assert_array_equal(got, ref_y)


def expert_out_dev(c: synth.Case, seed: int = 0):
    """Host stand-in expert outputs (valid rows filled) and the same bytes on
    the device; only the filled rows cross to the device."""
    eo = synth.make_expert_out(c, seed)
    v = c.topk_idx[(c.topk_idx >= 0) & (c.topk_idx < c.E)]
    cnt = np.bincount(v, minlength=c.E) if v.size else np.zeros(c.E, np.int64)
    rows = valid_rows(cnt, c.cap)
    dev = torch.zeros((c.E, c.cap, c.H), dtype=torch.bfloat16, device="cuda")
    if rows.size:
        flat = eo.reshape(c.E * c.cap, c.H)
        dev.view(c.E * c.cap, c.H)[torch.from_numpy(rows).cuda()] = bf16_dev(flat[rows])
    return eo, dev
