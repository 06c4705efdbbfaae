"""Seeded fuzz over random shapes through every GPU path, each checked against
the CPU oracle (bit-exact integers, rows, codes and scales; combine within
one bf16 ulp and bit-exact by construction), plus CUDA-graph replays of the
rank-major and e4m3 paths against eager runs."""
import numpy as np
import pytest
import torch

import oracle
from combine_moedc_layout_gb300 import moedc, synth
from parity_util import (DevCase, bf16_dev, bits_host, compare_combine, compare_dispatch,
                         compare_layout, expert_out_dev, run_layout, valid_rows)

pytestmark = pytest.mark.gpu


def _shape(seed):
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.choice([1, 2, 3, 4, 8, 16]))
    E = R * int(rng.integers(1, 33))
    K = int(rng.integers(1, min(E, 12) + 1))
    T = int(rng.choice([1, 2, 5, 17, 100, 333, 1500, 9000]))
    fp8 = bool(rng.integers(0, 2))
    H = 128 * int(rng.integers(1, 20)) if fp8 else 8 * int(rng.integers(1, 300))
    mask_p = float(rng.choice([0.0, 0.05, 0.5]))
    distinct = bool(rng.integers(0, 2)) and K <= E
    return dict(seed=seed, T=T, H=H, K=K, E=E, R=R, cap=None,
                dtype=synth.FP8_E4M3 if fp8 else synth.BF16, mask_p=mask_p, distinct=distinct)


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_layout_dispatch_combine(seed):
    c = synth.make_random_case(**_shape(seed))
    d = DevCase(c)
    fp8 = c.dtype == synth.FP8_E4M3
    if seed % 2:
        lay, recv, scales, src = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, c.dtype)
    else:
        lay = run_layout(d)
        recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, c.dtype)
    eo_host, eo = expert_out_dev(c, seed)
    y = moedc.combine(eo, d.topk_idx, lay.slot, d.topk_weights, status=lay.status)
    torch.cuda.synchronize()
    ref_lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    compare_layout(lay, ref_lay, c.T)
    ref_d = oracle.dispatch(c.x, c.topk_idx, ref_lay["slot"], c.E, c.cap, fp8=fp8)
    compare_dispatch(c, recv, scales, src, ref_lay, ref_d)
    compare_combine(y, oracle.combine(eo_host, c.topk_idx, ref_lay["slot"], c.topk_weights)["y"])
    if fp8:
        y8 = moedc.combine_e4m3(recv, scales, d.topk_idx, lay.slot, d.topk_weights)
        torch.cuda.synchronize()
        ref8 = oracle.combine_e4m3(ref_d["recv"], ref_d["scales"], c.topk_idx, ref_lay["slot"],
                                   c.topk_weights)
        compare_combine(y8, ref8["y"])


def _graph_vs_eager(fn, outs):
    """Run fn eagerly, snapshot outs, zero them, capture fn in a graph, replay
    twice, and require the same bytes."""
    fn(torch.cuda.current_stream())
    torch.cuda.synchronize()
    eager = [bits_host(t).copy() for t in outs]
    for t in outs:
        t.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn(s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, t in zip(eager, outs):
        np.testing.assert_array_equal(a, bits_host(t))


def test_graph_replay_rank_path_and_e4m3_combine():
    c = synth.make_case("default_ll")
    d = DevCase(c)
    lay = run_layout(d)
    torch.cuda.synchronize()
    ref_lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    cap_rank = int(ref_lay["num_tokens_per_rank"].max())
    dev = "cuda"
    rslot = torch.empty((c.T, c.R), dtype=torch.int32, device=dev)
    rrecv, rscales, rsrc = moedc.alloc_recv(c.R, cap_rank, c.H, c.dtype, dev)
    recv, scales, src = moedc.alloc_recv(c.E, c.cap, c.H, c.dtype, dev)
    y = torch.empty((c.T, c.H), dtype=torch.bfloat16, device=dev)
    yr = torch.empty((c.T, c.H), dtype=torch.bfloat16, device=dev)
    part = torch.zeros((c.R, cap_rank, c.H), dtype=torch.bfloat16, device=dev)
    part.view(-1)[: c.H * 3].fill_(0.5)

    def fn(s):
        assert moedc.moedc_rank_layout(lay.is_token_in_rank, c.T, c.R, cap_rank, rslot,
                                       lay.status, s) == moedc.OK
        assert moedc.moedc_rank_dispatch(d.x, c.T, c.H, rslot, lay.num_tokens_per_rank, c.R,
                                         cap_rank, c.dtype, rrecv, rscales, rsrc, s) == moedc.OK
        assert moedc.moedc_rank_combine(part, c.R, cap_rank, c.H, rslot, c.T, yr, s) == moedc.OK
        assert moedc.moedc_dispatch(d.x, c.T, c.H, d.topk_idx, lay.slot,
                                    lay.num_tokens_per_expert, c.K, c.E, c.cap, c.dtype, recv,
                                    scales, src, lay.status, s) == moedc.OK
        assert moedc.moedc_combine_e4m3(recv, scales, 0, c.E, c.cap, c.H, d.topk_idx, lay.slot,
                                        d.topk_weights, c.T, c.K, y, lay.status, s) == moedc.OK

    _graph_vs_eager(fn, [rslot, rsrc, yr, src, y])
    assert int(lay.status.item()) == 0


def _token_shape(seed):
    rng = np.random.default_rng(2000 + seed)
    R = int(rng.choice([1, 2, 4, 8]))
    E = R * int(rng.integers(1, 33))
    K = int(rng.integers(1, min(E, 10) + 1))
    T = int(rng.choice([1, 3, 40, 257, 2000]))
    H = 128 * int(rng.choice([1, 3, 5, 14, 56, 130, 256]))
    return dict(seed=seed, T=T, H=H, K=K, E=E, R=R, cap=None, dtype=synth.FP8_E4M3,
                mask_p=float(rng.choice([0.0, 0.1])), distinct=bool(rng.integers(0, 2)) and K <= E)


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_token_scale(seed):
    """Per-token e4m3 scales through dispatch, dequant and e4m3 combine."""
    c = synth.make_random_case(**_token_shape(seed))
    d = DevCase(c)
    tok = moedc.FP8_E4M3 | moedc.SCALES_PER_TOKEN
    if seed % 2:   # one call: a single launch up to 1024 entries
        lay, recv, scales, src = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, tok)
    else:
        lay = run_layout(d)
        recv, scales, src = moedc.dispatch(d.x, d.topk_idx, lay, c.E, c.cap, tok)
    deq = moedc.dequant_e4m3(recv, scales, lay.num_tokens_per_expert,
                             scale_layout=moedc.SCALES_PER_TOKEN)
    y = moedc.combine_e4m3(recv, scales, d.topk_idx, lay.slot, d.topk_weights,
                           scale_layout=moedc.SCALES_PER_TOKEN)
    torch.cuda.synchronize()
    ref_lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    ref = oracle.dispatch_token_scale(c.x, c.topk_idx, ref_lay["slot"], c.E, c.cap)
    compare_layout(lay, ref_lay, c.T)
    np.testing.assert_array_equal(src.cpu().numpy(), ref["src_idx"])
    rows = valid_rows(ref_lay["num_tokens_per_expert"], c.cap)
    if rows.size:
        ridx = torch.from_numpy(rows).cuda()
        np.testing.assert_array_equal(bits_host(recv.reshape(c.E * c.cap, c.H).index_select(0, ridx)),
                                      ref["recv"].reshape(c.E * c.cap, c.H)[rows])
        np.testing.assert_array_equal(scales.reshape(-1).index_select(0, ridx).cpu().numpy().view(np.uint32),
                                      ref["scales"].reshape(-1)[rows].view(np.uint32))
        ref_deq = oracle.dequant_e4m3_token(ref["recv"], ref["scales"], ref_lay["num_tokens_per_expert"])
        np.testing.assert_array_equal(bits_host(deq.reshape(c.E * c.cap, c.H).index_select(0, ridx)),
                                      ref_deq.reshape(c.E * c.cap, c.H)[rows])
    ref_y = oracle.combine_e4m3(ref["recv"], ref["scales"], c.topk_idx, ref_lay["slot"],
                                c.topk_weights, per_token=True)["y"]
    compare_combine(y, ref_y)


def _coop_shape(seed):
    rng = np.random.default_rng(3000 + seed)
    K = int(rng.choice([1, 4, 8, 16]))
    T = int(rng.integers(65536 // K + 1, 65536 // K + 30000))
    R = int(rng.choice([1, 2, 8, 16]))
    E = R * int(rng.integers(1, 17))
    K = min(K, E)
    T = max(T, 65536 // K + 1)
    fp8 = bool(rng.integers(0, 2))
    return dict(seed=seed, T=T, H=128 * int(rng.integers(1, 3)) if fp8 else 8 * int(rng.integers(2, 40)),
                K=K, E=E, R=R, cap=None, dtype=synth.FP8_E4M3 if fp8 else synth.BF16,
                mask_p=float(rng.choice([0.0, 0.03])), distinct=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_cooperative_layout_dispatch(seed):
    """Random shapes beyond 65536 routing entries through the one-call
    layout+dispatch, which runs as one cooperative launch there."""
    c = synth.make_random_case(**_coop_shape(seed))
    assert c.T * c.K > 65536
    d = DevCase(c)
    lay, recv, scales, src = moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, c.dtype)
    torch.cuda.synchronize()
    ref_lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    compare_layout(lay, ref_lay, c.T)
    ref_d = oracle.dispatch(c.x, c.topk_idx, ref_lay["slot"], c.E, c.cap,
                            fp8=c.dtype == synth.FP8_E4M3)
    compare_dispatch(c, recv, scales, src, ref_lay, ref_d)
