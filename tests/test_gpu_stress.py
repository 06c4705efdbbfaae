"""Many rounds and repeated runs on the GPU.

Rounds: 300 low-token rounds (16 tokens, hidden 6144, top-8 of 128, 16 ranks,
e4m3) with fresh seeded routing each round, through the single-launch
layout+dispatch and the combine, every round compared with the CPU oracle
and every status word clean - the many-rounds, zero-errors check that the
MORI pages run on their clusters.

Repeatability: the 4096-token step and the cooperative 40000-token launch
rerun on the same inputs must give the same bytes every time (several
kernels use shared-memory atomics, the status word and grid barriers, none
of which may change a result)."""
import numpy as np
import pytest
import torch

import oracle
from combine_moedc_layout_gb300 import moedc, synth
from parity_util import DevCase, compare_combine, compare_dispatch, compare_layout

pytestmark = pytest.mark.gpu


def test_300_low_token_rounds_against_the_oracle():
    base = synth.make_case("low16")
    for rnd in range(300):
        c = synth.make_case("low16", seed=1000 + rnd)
        assert (c.T, c.H, c.K, c.E) == (base.T, base.H, base.K, base.E)
        d = DevCase(c)
        lay, recv, scales, src = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, c.dtype)
        eo_host = synth.make_expert_out(c, rnd)
        eo = torch.from_numpy(eo_host.view(np.int16)).view(torch.bfloat16).cuda()
        y = moedc.combine(eo, d.topk_idx, lay.slot, d.topk_weights, status=lay.status)
        torch.cuda.synchronize()
        ref_lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
        compare_layout(lay, ref_lay, c.T)
        ref_d = oracle.dispatch(c.x, c.topk_idx, ref_lay["slot"], c.E, c.cap, fp8=True)
        compare_dispatch(c, recv, scales, src, ref_lay, ref_d)
        compare_combine(y, oracle.combine(eo_host, c.topk_idx, ref_lay["slot"],
                                          c.topk_weights)["y"])


def _snapshot(*ts):
    return [t.clone() for t in ts]


def _same(a, b):
    return all(torch.equal(x.view(torch.uint8) if x.dtype == torch.float8_e4m3fn else x,
                           y.view(torch.uint8) if y.dtype == torch.float8_e4m3fn else y)
               for x, y in zip(a, b))


def test_4096_token_step_repeats_bit_for_bit():
    c = synth.make_case("throughput")
    d = DevCase(c)
    g = torch.Generator(device="cuda").manual_seed(3)
    eo = torch.randn((c.E, c.cap, c.H), device="cuda", generator=g).to(torch.bfloat16)
    lay = moedc.layout(d.topk_idx, c.E, c.R, c.cap)
    recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, c.dtype)
    y = moedc.combine(eo, d.topk_idx, lay.slot, d.topk_weights, status=lay.status)
    torch.cuda.synchronize()
    cnt = lay.num_tokens_per_expert.cpu().numpy()
    rows = torch.from_numpy(np.concatenate([e * c.cap + np.arange(min(int(cnt[e]), c.cap))
                                            for e in range(c.E)])).cuda()

    def filled(t, width):
        return t.reshape(c.E * c.cap, width).index_select(0, rows)

    first = _snapshot(lay.slot, lay.num_tokens_per_expert, lay.num_tokens_per_rank,
                      lay.is_token_in_rank, src, filled(recv.view(torch.uint8), c.H),
                      filled(scales, c.G), y)
    for _ in range(40):
        lay2 = moedc.layout(d.topk_idx, c.E, c.R, c.cap, status=lay.status)
        moedc.dispatch(d.x, d.topk_idx, lay2, c.E, c.cap, c.dtype, out=(recv, scales, src))
        y2 = moedc.combine(eo, d.topk_idx, lay2.slot, d.topk_weights, status=lay.status)
        torch.cuda.synchronize()
        again = [lay2.slot, lay2.num_tokens_per_expert, lay2.num_tokens_per_rank,
                 lay2.is_token_in_rank, src, filled(recv.view(torch.uint8), c.H),
                 filled(scales, c.G), y2]
        assert _same(first, again)
    assert int(lay.status.item()) == 0


def test_cooperative_launch_repeats_bit_for_bit():
    c = synth.make_random_case(91, T=40000, H=128, K=8, E=128, R=8, cap=None, dtype=synth.BF16,
                               mask_p=0.01)
    d = DevCase(c)
    ws = moedc.layout_dispatch_workspace(c.T, c.K, c.E, c.R, "cuda")
    out = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, c.dtype, workspace=ws)
    torch.cuda.synchronize()
    lay, recv, _, src = out
    cnt = lay.num_tokens_per_expert.cpu().numpy()
    rows = torch.from_numpy(np.concatenate([e * c.cap + np.arange(min(int(cnt[e]), c.cap))
                                            for e in range(c.E)])).cuda()
    first = _snapshot(lay.slot, lay.num_tokens_per_expert, lay.num_tokens_per_rank,
                      lay.is_token_in_rank, src,
                      recv.reshape(c.E * c.cap, c.H).index_select(0, rows))
    for _ in range(40):
        lay2, recv2, _, src2 = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, c.dtype,
                                                     workspace=ws)
        torch.cuda.synchronize()
        assert int(lay2.status.item()) == 0
        assert _same(first, [lay2.slot, lay2.num_tokens_per_expert, lay2.num_tokens_per_rank,
                             lay2.is_token_in_rank, src2,
                             recv2.reshape(c.E * c.cap, c.H).index_select(0, rows)])
