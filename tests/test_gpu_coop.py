"""GPU parity of the cooperative single-launch layout + dispatch (T * K above
the single-launch layout's 65536 entries, workspace of
moedc_layout_dispatch_workspace_bytes):
against the CPU oracle, against the two-launch path on the same inputs, with
garbage in the workspace, under CUDA-graph replay, and the bounded barrier
wait running out (a test hook makes the barrier wait for one block too many)."""

import numpy as np
import pytest
import torch

import oracle
from combine_moedc_layout_gb300 import moedc, synth
from parity_util import DevCase, bits_host, compare_dispatch, compare_layout, valid_rows

pytestmark = pytest.mark.gpu

# every case has more than 65536 routing entries (the single-launch layout's
# limit), where moedc_layout_dispatch runs as one cooperative launch
CASES = {
    "t9000_fp8": lambda: synth.make_random_case(90, T=9000, H=1024, K=8, E=256, R=8, cap=None,
                                                dtype=synth.FP8_E4M3, mask_p=0.02),
    "large_t": lambda: synth.make_random_case(91, T=40000, H=128, K=8, E=128, R=8, cap=None,
                                              dtype=synth.BF16, mask_p=0.01),
    # more expert + rank rows (1032) than blocks
    "k32_e1024": lambda: synth.make_random_case(92, T=2100, H=256, K=32, E=1024, R=8, cap=None,
                                                dtype=synth.FP8_E4M3),
    "duplicates": lambda: synth.make_random_case(93, T=9000, H=256, K=8, E=5, R=5, cap=None,
                                                 dtype=synth.BF16, distinct=False),
    "k1": lambda: synth.make_random_case(94, T=70000, H=128, K=1, E=16, R=4, cap=None,
                                         dtype=synth.BF16),
    "e_eq_r": lambda: synth.make_random_case(95, T=17000, H=384, K=4, E=16, R=16, cap=None,
                                             dtype=synth.FP8_E4M3, mask_p=0.2),
    # 608 blocks on a GB300: 256-token chunks of exactly 2048 entries, the limit
    "max_chunk": lambda: synth.make_random_case(97, T=155648, H=128, K=8, E=128, R=8, cap=None,
                                                dtype=synth.BF16),
    # chunks over the limit: the call falls back to the two-launch layout
    "over_chunk": lambda: synth.make_random_case(98, T=200000, H=128, K=8, E=64, R=8, cap=None,
                                                 dtype=synth.BF16),
}

_cache = {}


def case(name):
    if name not in _cache:
        _cache[name] = CASES[name]()
    return _cache[name]


def _run(d, c, out_dtype, workspace):
    return moedc.layout_dispatch(d.x, d.topk_idx, c.E, c.R, c.cap, out_dtype,
                                 workspace=workspace)


def _coop_ws(c, fill=None):
    n = moedc.moedc_layout_dispatch_workspace_bytes(c.T, c.K, c.E, c.R)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    if fill is not None:
        ws.fill_(fill)
    return ws


def _oracle(c):
    lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    d = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap,
                        fp8=c.dtype == synth.FP8_E4M3)
    return lay, d


@pytest.mark.parametrize("name", list(CASES))
def test_coop_layout_dispatch_matches_oracle(name):
    c = case(name)
    d = DevCase(c)
    lay, recv, scales, src = _run(d, c, c.dtype, _coop_ws(c))
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle(c)
    compare_layout(lay, ref_lay, c.T)
    compare_dispatch(c, recv, scales, src, ref_lay, ref_d)


@pytest.mark.parametrize("name,cols", [("t9000_fp8", True), ("e_eq_r", False)])
def test_coop_equals_two_launch_path(name, cols):
    """Every output byte equal to layout then dispatch (two launches: the
    layout's own workspace is too small for the single launch)."""
    c = case(name)
    d = DevCase(c)
    dt = c.dtype | (moedc.SCALES_COL_MAJOR if cols else 0)
    a = _run(d, c, dt, _coop_ws(c, fill=0xFF))
    b = _run(d, c, dt, moedc.layout_workspace(c.T, c.K, c.E, c.R, "cuda"))
    torch.cuda.synchronize()
    la, lb = a[0], b[0]
    for f in ("num_tokens_per_expert", "num_tokens_per_rank", "is_token_in_rank", "slot",
              "status"):
        assert torch.equal(getattr(la, f), getattr(lb, f)), f
    assert torch.equal(a[3], b[3])
    rows = torch.from_numpy(valid_rows(la.num_tokens_per_expert.cpu().numpy(), c.cap)).cuda()
    np.testing.assert_array_equal(bits_host(a[1].reshape(c.E * c.cap, c.H).index_select(0, rows)),
                                  bits_host(b[1].reshape(c.E * c.cap, c.H).index_select(0, rows)))
    if c.dtype == synth.FP8_E4M3:            # scales of filled rows (the rest is not written)
        ga = a[2].cpu().numpy()
        gb = b[2].cpu().numpy()
        cnt = la.num_tokens_per_expert.cpu().numpy()
        for e in range(c.E):
            n = min(int(cnt[e]), c.cap)
            if cols:
                np.testing.assert_array_equal(ga[e, :, :n], gb[e, :, :n])
            else:
                np.testing.assert_array_equal(ga[e, :n], gb[e, :n])


@pytest.mark.parametrize("fill", [0x00, 0xFF, "random", "reuse"])
def test_coop_workspace_needs_no_initialisation(fill):
    c = case("t9000_fp8")
    d = DevCase(c)
    ws = _coop_ws(c)
    if fill == "random":
        ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda"))
    elif fill == "reuse":
        _run(d, c, c.dtype, ws)               # left by an earlier launch
    else:
        ws.fill_(fill)
    lay, recv, scales, src = _run(d, c, c.dtype, ws)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle(c)
    compare_layout(lay, ref_lay, c.T)
    compare_dispatch(c, recv, scales, src, ref_lay, ref_d)


def test_coop_status_capacity_and_range():
    c = synth.make_random_case(96, T=20000, H=256, K=4, E=8, R=2, cap=None, dtype=synth.BF16,
                               mask_p=0.1)
    c.cap = max(1, c.cap - 20)
    c.topk_idx[7, 2] = 9
    d = DevCase(c)
    lay, recv, scales, src = _run(d, c, c.dtype, _coop_ws(c))
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle(c)
    assert int(lay.status.item()) == oracle.ERR_EXPERT_RANGE == ref_lay["status"]
    compare_layout(lay, ref_lay, c.T)
    compare_dispatch(c, recv, scales, src, ref_lay, ref_d)


def test_coop_graph_replay_bit_exact():
    c = case("e_eq_r")
    d = DevCase(c)
    dev = "cuda"
    ws = _coop_ws(c)
    T, K, E, R, H, cap = c.T, c.K, c.E, c.R, c.H, c.cap
    cnt = torch.empty(E, dtype=torch.int32, device=dev)
    rk = torch.empty(R, dtype=torch.int32, device=dev)
    inr = torch.empty((T, R), dtype=torch.uint8, device=dev)
    sl = torch.empty((T, K), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    recv, scales, src = moedc.alloc_recv(E, cap, H, c.dtype, dev)

    def call(s):
        assert moedc.moedc_layout_dispatch(d.x, d.topk_idx, T, H, K, E, R, cap, c.dtype, cnt, rk,
                                           inr, sl, recv, scales, src, ws,
                                           ws.numel(), st, s) == moedc.OK

    call(torch.cuda.current_stream())
    torch.cuda.synchronize()
    eager = [t.clone() for t in (cnt, rk, inr, sl, src)]
    for t in (cnt, rk, inr, sl, src):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call(s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (cnt, rk, inr, sl, src)):
        assert torch.equal(a, b)
    assert int(st.item()) == 0


def test_coop_barrier_wait_runs_out_and_reports_timeout():
    """A barrier that waits for one block more than the grid has runs out of
    its bounded wait: the call reports MOEDC_ERR_TIMEOUT on the device status,
    the context stays usable, and the next call is correct."""
    c = case("t9000_fp8")
    d = DevCase(c)
    ws = _coop_ws(c)
    lib = moedc.load()
    lib.moedc_test_set_wait_extra(1)
    try:
        lay, *_ = _run(d, c, c.dtype, ws)
        torch.cuda.synchronize()
    finally:
        lib.moedc_test_set_wait_extra(0)
    assert int(lay.status.item()) == moedc.ERR_TIMEOUT
    lay, recv, scales, src = _run(d, c, c.dtype, ws)
    torch.cuda.synchronize()
    ref_lay, ref_d = _oracle(c)
    compare_layout(lay, ref_lay, c.T)
    compare_dispatch(c, recv, scales, src, ref_lay, ref_d)
