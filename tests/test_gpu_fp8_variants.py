"""GPU parity of the FP8 variants: column-major scale layout for dispatch and
dequant, and combine from e4m3 expert outputs, through the C ABI against the
CPU oracle.  Codes and scales bit-exact; combine within one bf16 ulp and, by
construction, bit-exact."""
import functools

import numpy as np
import pytest
import torch

import oracle
from combine_moedc_layout_gb300 import moedc, synth
from parity_util import DevCase, bits_host, compare_combine, run_layout, valid_rows

pytestmark = pytest.mark.gpu

CASES = {
    "low16": lambda: synth.make_case("low16"),
    "default_ll": lambda: synth.make_case("default_ll"),
    "throughput": lambda: synth.make_case("throughput"),
    "multiblock_fp8": lambda: synth.make_random_case(70, T=2500, H=1408, K=8, E=64, R=8,
                                                     cap=None, dtype=synth.FP8_E4M3,
                                                     mask_p=0.03),
    "k20": lambda: synth.make_random_case(72, T=300, H=384, K=20, E=40, R=4, cap=None,
                                          dtype=synth.FP8_E4M3, mask_p=0.1),
}


@functools.lru_cache(maxsize=None)
def case(name):
    return CASES[name]()


def _oracle_chain(c):
    lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=True)
    return lay, d


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("fused", [False, True])
def test_column_major_scales(name, fused):
    c = case(name)
    d = DevCase(c)
    dtype = moedc.FP8_E4M3 | moedc.SCALES_COL_MAJOR
    if fused:
        lay, recv, scales, src = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, dtype)
    else:
        lay = run_layout(d)
        recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, dtype)
    assert tuple(scales.shape) == (c.E, c.G, c.cap)
    deq_cols = moedc.dequant_e4m3(recv, scales, lay.num_tokens_per_expert,
                                  scale_layout=moedc.SCALES_COL_MAJOR)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle_chain(c)
    np.testing.assert_array_equal(src.cpu().numpy(), ref_d["src_idx"])
    cnt = ref_lay["num_tokens_per_expert"]
    rows = valid_rows(cnt, c.cap)
    ridx = torch.from_numpy(rows).cuda()
    got = bits_host(recv.reshape(c.E * c.cap, c.H).index_select(0, ridx))
    np.testing.assert_array_equal(got, ref_d["recv"].reshape(c.E * c.cap, c.H)[rows])
    gs = scales.cpu().numpy()                                   # [E, G, cap]
    ws = ref_d["scales"].transpose(0, 2, 1)                     # [E, G, cap]
    for e in range(c.E):
        n = min(cnt[e], c.cap)
        np.testing.assert_array_equal(gs[e, :, :n].view(np.uint32), ws[e, :, :n].view(np.uint32))
    ref_deq = oracle.dequant_e4m3(ref_d["recv"], ref_d["scales"], cnt)
    gd = bits_host(deq_cols.reshape(c.E * c.cap, c.H).index_select(0, ridx))
    np.testing.assert_array_equal(gd, ref_deq.reshape(c.E * c.cap, c.H)[rows])


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("cols", [False, True])
def test_combine_e4m3_parity(name, cols):
    """Identity experts: the e4m3 rows dispatch wrote are the expert outputs."""
    c = case(name)
    d = DevCase(c)
    dtype = moedc.FP8_E4M3 | (moedc.SCALES_COL_MAJOR if cols else 0)
    lay = run_layout(d)
    recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, dtype)
    y = moedc.combine_e4m3(recv, scales, d.topk_idx, lay.slot, d.topk_weights,
                           scale_layout=moedc.SCALES_COL_MAJOR if cols else 0,
                           status=lay.status)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle_chain(c)
    ref = oracle.combine_e4m3(ref_d["recv"], ref_d["scales"], c.topk_idx, ref_lay["slot"],
                              c.topk_weights)
    assert int(lay.status.item()) == ref["status"] == 0
    compare_combine(y, ref["y"])


def test_combine_e4m3_skips_masked_out_of_range_and_dropped():
    c = synth.make_random_case(73, T=500, H=256, K=4, E=8, R=2, cap=None, dtype=synth.FP8_E4M3,
                               mask_p=0.15)
    c.cap = max(1, c.cap - 10)                  # drop the last entries of the fullest experts
    c.topk_idx[3, 2] = 8                         # out of range
    d = DevCase(c)
    lay = run_layout(d)
    recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, moedc.FP8_E4M3)
    y = moedc.combine_e4m3(recv, scales, d.topk_idx, lay.slot, d.topk_weights, status=lay.status)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle_chain(c)
    ref = oracle.combine_e4m3(ref_d["recv"], ref_d["scales"], c.topk_idx, ref_lay["slot"],
                              c.topk_weights)
    assert int(lay.status.item()) == oracle.ERR_EXPERT_RANGE
    compare_combine(y, ref["y"])
