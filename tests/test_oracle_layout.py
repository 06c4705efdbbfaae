"""Pins for the oracle's routing layout.

References independent of the oracle: a hand-worked fixture, exhaustive
enumeration of tiny routing matrices checked against a sort-based
formulation (a stable sort of (expert, token, k) triples gives each expert's
slot order directly), and invariants that must hold at any size.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from combine_moedc_layout_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sorted_layout(idx: np.ndarray, E: int, R: int):
    """Layout through a stable sort: a different formulation from the oracle's
    single counting pass."""
    T, K = idx.shape
    epr = E // R
    flat = idx.reshape(-1)
    pos = np.arange(flat.size)
    live = (flat >= 0) & (flat < E)
    # sort key: expert first, then flat position (= token, then k)
    order = np.lexsort((pos[live], flat[live]))
    experts = flat[live][order]
    where = pos[live][order]
    slot = np.full(flat.size, -1, np.int64)
    counts = np.zeros(E, np.int64)
    start = 0
    for e in range(E):
        n = int((experts == e).sum())
        slot[where[start:start + n]] = np.arange(n)
        counts[e] = n
        start += n
    in_rank = np.zeros((T, R), np.uint8)
    for t in range(T):
        for e in set(int(v) for v in idx[t] if 0 <= v < E):
            in_rank[t, e // epr] = 1
    return counts, in_rank.sum(axis=0), in_rank, slot.reshape(T, K)


def test_golden_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "layout_t4_k2_e4_r2.json")))
    idx = np.array(g["topk_idx"], np.int32)
    out = oracle.layout(idx, g["E"], g["R"], g["cap"])
    np.testing.assert_array_equal(out["num_tokens_per_expert"], g["num_tokens_per_expert"])
    np.testing.assert_array_equal(out["num_tokens_per_rank"], g["num_tokens_per_rank"])
    np.testing.assert_array_equal(out["is_token_in_rank"], g["is_token_in_rank"])
    np.testing.assert_array_equal(out["slot"], g["slot"])
    assert out["status"] == g["status"]
    assert oracle.layout(idx, g["E"], g["R"], 2)["status"] == g["status_with_cap_2"]
    # src_idx comes out of dispatch
    x = np.zeros((g["T"], 128), np.uint16)
    d = oracle.dispatch(x, idx, out["slot"], g["E"], g["cap"], fp8=False)
    np.testing.assert_array_equal(d["src_idx"], g["src_idx"])


@pytest.mark.parametrize("T,K,E,R", [(2, 2, 2, 1), (2, 2, 2, 2), (3, 2, 3, 3), (2, 3, 2, 2),
                                     (3, 1, 4, 2), (1, 4, 3, 1)])
def test_exhaustive_tiny(T, K, E, R):
    vals = range(-1, E)
    n = 0
    for combo in itertools.product(vals, repeat=T * K):
        idx = np.array(combo, np.int32).reshape(T, K)
        out = oracle.layout(idx, E, R, cap=T * K)
        cnt, per_rank, in_rank, slot = _sorted_layout(idx, E, R)
        np.testing.assert_array_equal(out["num_tokens_per_expert"], cnt)
        np.testing.assert_array_equal(out["num_tokens_per_rank"], per_rank)
        np.testing.assert_array_equal(out["is_token_in_rank"], in_rank)
        np.testing.assert_array_equal(out["slot"], slot)
        assert out["status"] == oracle.OK
        n += 1
    assert n == (E + 1) ** (T * K)


def _check_invariants(idx, E, R, cap, out):
    T, K = idx.shape
    live = (idx >= 0) & (idx < E)
    cnt = out["num_tokens_per_expert"]
    slot = out["slot"]
    assert int(cnt.sum()) == int(live.sum())                      # counts sum to N
    assert (slot[~live] == -1).all()
    for e in range(E):
        t_of, k_of = np.nonzero(idx == e)
        s = slot[t_of, k_of]
        np.testing.assert_array_equal(np.sort(s), np.arange(cnt[e]))  # a permutation
        order = np.lexsort((k_of, t_of))
        assert (np.diff(s[order]) == 1).all()                     # ascending token order
    any_live = live.any(axis=1).sum()
    assert int(out["num_tokens_per_rank"].sum()) >= int(any_live)
    assert (out["num_tokens_per_rank"] <= T).all()
    d = oracle.dispatch(np.zeros((T, 128), np.uint16), idx, slot, E, cap, fp8=False)
    src = d["src_idx"]
    for t, k in zip(*np.nonzero(live)):                           # src_idx inverts slot
        if slot[t, k] < cap:
            assert src[idx[t, k], slot[t, k]] == t
    filled = (src >= 0).sum(axis=1)
    np.testing.assert_array_equal(filled, np.minimum(cnt, cap))


@pytest.mark.parametrize("name", ["tiny", "low16", "default_ll"])
def test_invariants_named_workloads(name):
    c = synth.make_case(name)
    out = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    assert out["status"] == oracle.OK
    _check_invariants(c.topk_idx, c.E, c.R, c.cap, out)
    cnt, per_rank, in_rank, slot = _sorted_layout(c.topk_idx, c.E, c.R)
    np.testing.assert_array_equal(out["slot"], slot)
    np.testing.assert_array_equal(out["num_tokens_per_rank"], per_rank)


def test_invariants_duplicates_allowed():
    c = synth.make_random_case(3, T=50, H=128, K=6, E=5, R=5, cap=None, dtype=synth.BF16,
                               mask_p=0.2, distinct=False)
    out = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    assert out["status"] == oracle.OK
    _check_invariants(c.topk_idx, c.E, c.R, c.cap, out)


def test_capacity_and_range_status():
    idx = np.array([[0, 1], [0, 1], [0, -1]], np.int32)
    assert oracle.layout(idx, 2, 1, cap=3)["status"] == oracle.OK
    out = oracle.layout(idx, 2, 1, cap=2)
    assert out["status"] == oracle.ERR_CAPACITY
    np.testing.assert_array_equal(out["slot"][:, 0], [0, 1, 2])   # slots keep counting
    bad = np.array([[0, 2], [-2, 1]], np.int32)
    out = oracle.layout(bad, 2, 2, cap=4)
    assert out["status"] == oracle.ERR_EXPERT_RANGE
    np.testing.assert_array_equal(out["slot"], [[0, -1], [-1, 0]])
    np.testing.assert_array_equal(out["num_tokens_per_expert"], [1, 1])
    # both problems: the larger code is reported
    both = np.array([[0, 5], [0, 0]], np.int32)
    assert oracle.layout(both, 2, 1, cap=1)["status"] == oracle.ERR_EXPERT_RANGE


def test_imbalanced_workload_shape():
    c = synth.make_case("imbalanced")
    live = c.topk_idx[c.topk_idx >= 0]
    load = np.bincount(live // (c.E // c.R), minlength=c.R)
    assert abs(load[0] / load.mean() - 1.5) <= 0.02
    assert abs((c.topk_idx < 0).mean() - 0.10) < 0.01
    out = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    assert out["status"] == oracle.OK
    assert int(out["num_tokens_per_expert"].max()) == c.cap
