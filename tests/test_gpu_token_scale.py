"""GPU parity of the per-token e4m3 variants through the C ABI: dispatch with
one scale per token row (scales [E, cap]), its dequantisation, and combine
from e4m3 rows with per-row scales, against the CPU oracle.  Codes, scales,
src_idx and dequantised rows bit-exact; combine within one bf16 ulp and, by
construction, bit-exact."""
import functools

import numpy as np
import pytest
import torch

import oracle
from combine_moedc_layout_gb300 import moedc, synth
from parity_util import DevCase, bits_host, compare_combine, compare_layout, run_layout, valid_rows

pytestmark = pytest.mark.gpu

TOK = moedc.FP8_E4M3 | moedc.SCALES_PER_TOKEN

CASES = {
    "low4": lambda: synth.make_case("low4"),
    "low16": lambda: synth.make_case("low16"),
    "default_ll": lambda: synth.make_case("default_ll"),
    "throughput": lambda: synth.make_case("throughput"),
    # one slice (one warp per block), a partial last slice, two and four slices per warp
    "h128": lambda: synth.make_random_case(80, T=300, H=128, K=4, E=16, R=4, cap=None,
                                           dtype=synth.FP8_E4M3, mask_p=0.05),
    "h640": lambda: synth.make_random_case(81, T=257, H=640, K=6, E=24, R=6, cap=None,
                                           dtype=synth.FP8_E4M3, mask_p=0.1),
    "h12288": lambda: synth.make_random_case(82, T=70, H=12288, K=8, E=32, R=4, cap=None,
                                             dtype=synth.FP8_E4M3),
    "h32768": lambda: synth.make_random_case(83, T=20, H=32768, K=4, E=8, R=2, cap=None,
                                             dtype=synth.FP8_E4M3),
    "duplicates": lambda: synth.make_random_case(84, T=500, H=1024, K=8, E=5, R=5, cap=None,
                                                 dtype=synth.FP8_E4M3, distinct=False),
    "tiny_values": lambda: synth.make_random_case(85, T=64, H=256, K=4, E=8, R=2, cap=None,
                                                  dtype=synth.FP8_E4M3, scale=1e-30),
}


@functools.lru_cache(maxsize=None)
def case(name):
    return CASES[name]()


def _oracle(c):
    lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    d = oracle.dispatch_token_scale(c.x, c.topk_idx, lay["slot"], c.E, c.cap)
    return lay, d


def _compare(c, recv, scales, src, ref_lay, ref_d):
    assert tuple(scales.shape) == (c.E, c.cap)
    np.testing.assert_array_equal(src.cpu().numpy(), ref_d["src_idx"])
    rows = valid_rows(ref_lay["num_tokens_per_expert"], c.cap)
    if rows.size == 0:
        return
    ridx = torch.from_numpy(rows).cuda()
    got = bits_host(recv.reshape(c.E * c.cap, c.H).index_select(0, ridx))
    np.testing.assert_array_equal(got, ref_d["recv"].reshape(c.E * c.cap, c.H)[rows])
    gs = scales.reshape(-1).index_select(0, ridx).cpu().numpy()
    np.testing.assert_array_equal(gs.view(np.uint32),
                                  ref_d["scales"].reshape(-1)[rows].view(np.uint32))


@pytest.mark.parametrize("name", list(CASES))
def test_dispatch_token_scale_parity(name):
    c = case(name)
    d = DevCase(c)
    lay = run_layout(d)
    recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, TOK)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle(c)
    assert int(lay.status.item()) == ref_d["status"] == 0
    _compare(c, recv, scales, src, ref_lay, ref_d)


@pytest.mark.parametrize("name", list(CASES))
def test_layout_dispatch_token_scale_parity(name):
    """The one-call entry point: a single launch whose blocks own whole tokens
    up to 1024 routing entries (low4, low16, default_ll, h12288, h32768,
    tiny_values: one, two and four slices per warp), layout then dispatch
    beyond."""
    c = case(name)
    d = DevCase(c)
    lay, recv, scales, src = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, TOK)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle(c)
    compare_layout(lay, ref_lay, c.T)
    _compare(c, recv, scales, src, ref_lay, ref_d)


@pytest.mark.parametrize("name", ["low16", "default_ll", "h12288", "duplicates"])
def test_dequant_and_combine_e4m3_per_token(name):
    c = case(name)
    d = DevCase(c)
    lay = run_layout(d)
    recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, TOK)
    deq = moedc.dequant_e4m3(recv, scales, lay.num_tokens_per_expert,
                             scale_layout=moedc.SCALES_PER_TOKEN)
    y = moedc.combine_e4m3(recv, scales, d.topk_idx, lay.slot, d.topk_weights,
                           scale_layout=moedc.SCALES_PER_TOKEN, status=lay.status)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle(c)
    cnt = ref_lay["num_tokens_per_expert"]
    rows = valid_rows(cnt, c.cap)
    ref_deq = oracle.dequant_e4m3_token(ref_d["recv"], ref_d["scales"], cnt)
    got = bits_host(deq.reshape(c.E * c.cap, c.H).index_select(0, torch.from_numpy(rows).cuda()))
    np.testing.assert_array_equal(got, ref_deq.reshape(c.E * c.cap, c.H)[rows])
    ref = oracle.combine_e4m3(ref_d["recv"], ref_d["scales"], c.topk_idx, ref_lay["slot"],
                              c.topk_weights, per_token=True)
    assert int(lay.status.item()) == ref["status"] == 0
    compare_combine(y, ref["y"])


def test_token_scale_drops_masks_and_flags_out_of_range():
    c = synth.make_random_case(86, T=400, H=768, K=4, E=8, R=2, cap=None, dtype=synth.FP8_E4M3,
                               mask_p=0.15)
    c.cap = max(1, c.cap - 12)                 # the fullest experts drop their last entries
    c.topk_idx[5, 1] = 8                       # out of range
    d = DevCase(c)
    lay = run_layout(d)
    recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, TOK)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle(c)
    assert int(lay.status.item()) == oracle.ERR_EXPERT_RANGE
    assert ref_d["status"] == oracle.ERR_EXPERT_RANGE
    _compare(c, recv, scales, src, ref_lay, ref_d)


def test_single_launch_token_scale_drops_masks_and_flags_out_of_range():
    """The same data errors through the one-call single launch (400 entries)."""
    c = synth.make_random_case(87, T=100, H=640, K=4, E=8, R=4, cap=None, dtype=synth.FP8_E4M3,
                               mask_p=0.15)
    c.cap = max(1, c.cap - 5)
    c.topk_idx[9, 3] = 11
    d = DevCase(c)
    lay, recv, scales, src = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, TOK)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle(c)
    assert ref_lay["status"] == oracle.ERR_EXPERT_RANGE
    compare_layout(lay, ref_lay, c.T)
    _compare(c, recv, scales, src, ref_lay, ref_d)


@pytest.mark.parametrize("one_call", [False, True])
def test_token_scale_empty_and_all_masked(one_call):
    """T = 0, and every entry masked: nothing is written but src_idx = -1
    everywhere and zero counts; no data error."""
    for T, mask in ((0, 0.0), (37, 1.0)):
        c = synth.make_random_case(88, T=T, H=384, K=4, E=8, R=2, cap=5, dtype=synth.FP8_E4M3,
                                   mask_p=mask)
        d = DevCase(c)
        if one_call:
            lay, recv, scales, src = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, TOK)
        else:
            lay = run_layout(d)
            recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, TOK)
        torch.cuda.synchronize()
        assert int(lay.status.item()) == 0
        assert (lay.num_tokens_per_expert.cpu().numpy() == 0).all()
        assert (lay.num_tokens_per_rank.cpu().numpy() == 0).all()
        assert (src.cpu().numpy() == -1).all()
