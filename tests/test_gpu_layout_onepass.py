"""GPU parity of the two one-launch layouts for up to 65536 routing entries:
the single-pass layout (with a workspace) and the sweep (without one), each
against the CPU oracle bit for bit, plus the single-pass layout's workspace
rules: any initial contents, reuse across shapes, replays of a captured graph
with new routing, and a bounded wait that runs out (MOEDC_ERR_TIMEOUT, after
which the next call is correct)."""
import numpy as np
import pytest
import torch

import oracle
from combine_moedc_layout_gb300 import moedc, synth
from parity_util import DevCase, compare_layout

pytestmark = pytest.mark.gpu

NAMED = ["tiny", "low4", "low16", "default_ll", "throughput", "imbalanced"]
RANDOM = {
    "multichunk_k6": dict(seed=31, T=3001, H=8, K=6, E=96, R=12, cap=None, dtype=synth.BF16,
                          mask_p=0.07),
    "k1": dict(seed=32, T=9000, H=8, K=1, E=16, R=4, cap=None, dtype=synth.BF16),
    "k32_e1024": dict(seed=33, T=2048, H=8, K=32, E=1024, R=8, cap=None, dtype=synth.BF16),
    "e_eq_r_1024": dict(seed=34, T=600, H=8, K=8, E=1024, R=1024, cap=None, dtype=synth.BF16,
                        mask_p=0.02),
    "one_expert": dict(seed=35, T=5000, H=8, K=1, E=1, R=1, cap=None, dtype=synth.BF16),
    "duplicates": dict(seed=36, T=900, H=8, K=8, E=5, R=5, cap=None, dtype=synth.BF16,
                       distinct=False),
    "t1": dict(seed=37, T=1, H=8, K=8, E=256, R=8, cap=1, dtype=synth.BF16),
    "max_entries": dict(seed=38, T=8192, H=8, K=8, E=256, R=8, cap=None, dtype=synth.BF16,
                        mask_p=0.1),
    "chunk_edge": dict(seed=39, T=129, H=8, K=8, E=64, R=8, cap=None, dtype=synth.BF16),
    "four_chunks": dict(seed=41, T=512, H=8, K=8, E=64, R=8, cap=None, dtype=synth.BF16,
                        mask_p=0.05),
    "four_chunks_ragged": dict(seed=42, T=450, H=8, K=8, E=24, R=3, cap=None,
                               dtype=synth.BF16),
    "k3_ragged": dict(seed=40, T=21845, H=8, K=3, E=48, R=6, cap=None, dtype=synth.BF16,
                      mask_p=0.3),
    # token-in-rank from shuffles (K a power of two, R <= K): one rank, fewer
    # ranks than K, two entries per token with repeats
    "k4_r1": dict(seed=43, T=3000, H=8, K=4, E=12, R=1, cap=None, dtype=synth.BF16, mask_p=0.1),
    "k16_r4": dict(seed=44, T=2000, H=8, K=16, E=64, R=4, cap=None, dtype=synth.BF16,
                   mask_p=0.05),
    "k2_r2": dict(seed=45, T=9000, H=8, K=2, E=10, R=2, cap=None, dtype=synth.BF16,
                  distinct=False),
    # more ranks than K, in rounds of K ranks: EP16 with top-8, 32 ranks with K = 4 and K = 2
    "k8_r16": dict(seed=46, T=3000, H=8, K=8, E=128, R=16, cap=None, dtype=synth.BF16,
                   mask_p=0.05),
    "k4_r32": dict(seed=47, T=5000, H=8, K=4, E=64, R=32, cap=None, dtype=synth.BF16),
    "k2_r32": dict(seed=48, T=7000, H=8, K=2, E=96, R=32, cap=None, dtype=synth.BF16,
                   distinct=False, mask_p=0.1),
}


def _case(key):
    return synth.make_case(key) if key in NAMED else synth.make_random_case(**RANDOM[key])


def _chunks(c):
    return max(1, -(-c.T // (1024 // c.K)))


# the single-pass layout runs from 4 chunks of 1024 entries; below, the sweep
SMALL = ["tiny", "low4", "low16", "default_ll", "t1", "chunk_edge"]
ONEPASS = [k for k in NAMED + list(RANDOM) if k not in SMALL]


def _outputs(T, K, E, R):
    dev = "cuda"
    return dict(cnt=torch.full((E,), -7, dtype=torch.int32, device=dev),
                rk=torch.full((R,), -7, dtype=torch.int32, device=dev),
                inr=torch.full((T, R), 9, dtype=torch.uint8, device=dev),
                slot=torch.full((T, K), -7, dtype=torch.int32, device=dev),
                st=torch.zeros(1, dtype=torch.int32, device=dev))


class _Lay:
    def __init__(self, o):
        self.num_tokens_per_expert = o["cnt"]
        self.num_tokens_per_rank = o["rk"]
        self.is_token_in_rank = o["inr"]
        self.slot = o["slot"]
        self.status = o["st"]


def _run(idx, c, ws, stream=None):
    o = _outputs(c.T, c.K, c.E, c.R)
    wsb = 0 if ws is None else ws.numel()
    rc = moedc.moedc_layout(idx, c.T, c.K, c.E, c.R, c.cap, o["cnt"], o["rk"], o["inr"],
                            o["slot"], ws, wsb, o["st"], stream)
    assert rc == moedc.OK
    return o


def _check(o, c):
    torch.cuda.synchronize()
    ref = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    compare_layout(_Lay(o), ref, c.T)
    assert int(o["st"].item()) == ref["status"]


@pytest.mark.parametrize("key", [pytest.param(k, id="onepass-" + k) for k in ONEPASS] +
                         [pytest.param(k, id="sweep-" + k) for k in NAMED + list(RANDOM)])
def test_layout_paths_match_oracle(request, key):
    c = _case(key)
    assert c.T * c.K <= 65536
    d = DevCase(c)
    ws = None
    if request.node.callspec.id.startswith("onepass"):
        n = moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R)
        assert _chunks(c) >= 4 and n > 0
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    _check(_run(d.topk_idx, c, ws), c)


@pytest.mark.parametrize("key", SMALL)
def test_small_shapes_take_the_sweep_and_ignore_a_workspace(key):
    """Below 4 chunks the size query is 0 and a workspace passed anyway
    changes nothing: the sweep runs and the results are the oracle's."""
    c = _case(key)
    assert _chunks(c) < 4
    assert moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R) == 0
    d = DevCase(c)
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    _check(_run(d.topk_idx, c, ws), c)


@pytest.mark.parametrize("fill", ["zeros", "ones", "random"])
def test_onepass_any_workspace_contents(fill):
    c = _case("throughput")
    d = DevCase(c)
    n = moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R)
    if fill == "zeros":
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    elif fill == "ones":
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    else:
        g = torch.Generator(device="cuda").manual_seed(5)
        ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
    _check(_run(d.topk_idx, c, ws), c)


def test_onepass_workspace_reused_across_shapes_and_routings():
    # one workspace, large enough for the largest shape, calls back to back
    keys = ["max_entries", "tiny", "throughput", "k32_e1024", "t1", "multichunk_k6", "throughput"]
    cases = [_case(k) for k in keys]
    n = max(moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R) for c in cases)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    outs = []
    for c in cases:
        outs.append((c, _run(DevCase(c).topk_idx, c, ws)))
    for c, o in outs:
        _check(o, c)


def test_onepass_graph_replays_with_new_routing():
    """Replays of one captured call share the host epoch; the workspace's
    generation must still keep one replay's flags from releasing the next."""
    base = _case("throughput")
    T, K, E, R = base.T, base.K, base.E, base.R
    idx = torch.from_numpy(base.topk_idx).cuda()
    n = moedc.moedc_layout_workspace_bytes(T, K, E, R)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    o = _outputs(T, K, E, R)

    def call(stream):
        assert moedc.moedc_layout(idx, T, K, E, R, base.cap, o["cnt"], o["rk"], o["inr"],
                                  o["slot"], ws, n, o["st"], stream) == moedc.OK

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)                                   # warm-up outside the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call(s)
    torch.cuda.synchronize()
    for seed in (50, 51, 52):
        c = synth.make_random_case(seed, T=T, H=8, K=K, E=E, R=R, cap=None, dtype=synth.BF16,
                                   mask_p=0.05)
        c.cap = base.cap            # the captured call's cap
        idx.copy_(torch.from_numpy(c.topk_idx))
        o["st"].zero_()
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.layout(c.topk_idx, E, R, base.cap)
        compare_layout(_Lay(o), ref, T)
        assert int(o["st"].item()) == ref["status"]


@pytest.mark.parametrize("key", ["throughput", "four_chunks"])
def test_onepass_wait_runs_out_and_reports_timeout(key):
    """A bounded wait of the single-pass layout that runs out raises
    MOEDC_ERR_TIMEOUT (the test hook makes the last block wait for a flag no
    block writes), the context stays usable and the next call is correct."""
    c = _case(key)
    d = DevCase(c)
    n = moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    lib = moedc.load()
    lib.moedc_test_set_wait_extra(1)
    try:
        o = _run(d.topk_idx, c, ws)
        torch.cuda.synchronize()
    finally:
        lib.moedc_test_set_wait_extra(0)
    assert int(o["st"].item()) == moedc.ERR_TIMEOUT
    _check(_run(d.topk_idx, c, ws), c)


def _status_case(kind):
    c = synth.make_random_case(60, T=2000, H=8, K=6, E=24, R=4, cap=None, dtype=synth.BF16,
                               mask_p=0.03)
    assert _chunks(c) >= 4
    if kind in ("capacity", "both"):
        c.cap = max(1, c.cap - 15)                 # the fullest experts overflow
    if kind in ("range", "both"):
        c.topk_idx[0, 2] = c.E                     # first chunk
        c.topk_idx[c.T // 2, 0] = -9               # a middle chunk
        c.topk_idx[c.T - 1, c.K - 1] = 10 ** 6     # the last chunk
    return c


@pytest.mark.parametrize("kind", ["capacity", "range", "both"])
@pytest.mark.parametrize("path", ["onepass", "sweep"])
def test_status_codes_match_oracle(kind, path):
    """Capacity overflow and out-of-range ids spread over several chunks: the
    device status is the oracle's (the larger code when both occur), counts
    keep counting past cap, and out-of-range entries get slot -1."""
    c = _status_case(kind)
    d = DevCase(c)
    ws = None
    if path == "onepass":
        ws = torch.empty(moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R), dtype=torch.uint8,
                         device="cuda")
    o = _run(d.topk_idx, c, ws)
    ref = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    expect = {"capacity": oracle.ERR_CAPACITY, "range": oracle.ERR_EXPERT_RANGE,
              "both": oracle.ERR_EXPERT_RANGE}[kind]
    assert ref["status"] == expect
    _check(o, c)


# beyond 65536 entries: the single pass at 1, 2 and 4 entries per thread, and
# the two-kernel layout (given exactly its own workspace) on the same shapes
LARGE = {
    "ept1_96000": dict(seed=70, T=12000, H=8, K=8, E=256, R=8, cap=None, dtype=synth.BF16,
                       mask_p=0.02),
    "ept2_160000": dict(seed=71, T=20000, H=8, K=8, E=128, R=8, cap=None, dtype=synth.BF16),
    "ept4_320000": dict(seed=72, T=40000, H=8, K=8, E=128, R=8, cap=None, dtype=synth.BF16,
                        mask_p=0.01),
    "ept4_540000": dict(seed=73, T=90000, H=8, K=6, E=60, R=6, cap=None, dtype=synth.BF16,
                        mask_p=0.05),
    "beyond_720000": dict(seed=74, T=120000, H=8, K=6, E=60, R=6, cap=None, dtype=synth.BF16),
    "ept2_k2_160000": dict(seed=75, T=80000, H=8, K=2, E=10, R=2, cap=None, dtype=synth.BF16,
                           mask_p=0.05),
    "ept2_r16_160000": dict(seed=76, T=20000, H=8, K=8, E=128, R=16, cap=None,
                            dtype=synth.BF16),
}


def _blocked_bytes(T, K, E, R):
    tpc = max(-(-1024 // K), -(-T // 1024))
    return -(-T // tpc) * (E + R) * 4


@pytest.mark.parametrize("key", list(LARGE))
@pytest.mark.parametrize("ws_size", ["query", "two_kernel"])
def test_large_layouts_match_oracle(key, ws_size):
    """With the queried workspace the single pass runs (the two-kernel layout
    beyond 144 chunks); with exactly the two-kernel layout's size that layout
    runs wherever it needs less than the single pass (96000 and 160000
    entries here)."""
    c = synth.make_random_case(**LARGE[key])
    assert c.T * c.K > 65536
    d = DevCase(c)
    n = moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R) if ws_size == "query" else \
        _blocked_bytes(c.T, c.K, c.E, c.R)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    _check(_run(d.topk_idx, c, ws), c)


def test_large_single_pass_wait_runs_out_and_reports_timeout():
    c = synth.make_random_case(**LARGE["ept4_320000"])
    d = DevCase(c)
    ws = torch.empty(moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R), dtype=torch.uint8,
                     device="cuda")
    lib = moedc.load()
    lib.moedc_test_set_wait_extra(1)
    try:
        o = _run(d.topk_idx, c, ws)
        torch.cuda.synchronize()
    finally:
        lib.moedc_test_set_wait_extra(0)
    assert int(o["st"].item()) == moedc.ERR_TIMEOUT
    _check(_run(d.topk_idx, c, ws), c)


def test_single_pass_fuzz_back_to_back_on_one_workspace():
    """40 random shapes (1, 2 and 4 entries per thread, 4 to 144 chunks, masks,
    duplicates, skewed expert counts) run back to back on one workspace that
    is never cleared, each checked against the oracle: every call must see
    only its own epoch's words, whatever the earlier calls left."""
    rng = np.random.default_rng(2024)
    shapes = []
    for i in range(40):
        R = int(rng.choice([1, 2, 4, 8, 16]))
        E = R * int(rng.integers(1, 33))
        K = int(rng.integers(1, min(E, 10) + 1))
        n = int(rng.integers(3073, 560000))
        T = max(1, n // K)
        shapes.append(dict(seed=500 + i, T=T, H=8, K=K, E=E, R=R, cap=None, dtype=synth.BF16,
                           mask_p=float(rng.choice([0.0, 0.1])),
                           distinct=bool(rng.integers(0, 2)) and K <= E))
    cases = [synth.make_random_case(**sh) for sh in shapes]
    sizes = [moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R) for c in cases]
    ws = torch.empty(max(sizes), dtype=torch.uint8, device="cuda")
    ran_single_pass = 0
    for c, n in zip(cases, sizes):
        o = _outputs(c.T, c.K, c.E, c.R)
        idx = torch.from_numpy(c.topk_idx).cuda()
        assert moedc.moedc_layout(idx, c.T, c.K, c.E, c.R, c.cap, o["cnt"], o["rk"], o["inr"],
                                  o["slot"], ws, ws.numel(), o["st"]) == moedc.OK
        _check(o, c)
        ran_single_pass += 1 if n > 0 else 0
    assert ran_single_pass >= 30
