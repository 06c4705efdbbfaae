"""Pins for the oracle's rank-major packed receive (a token goes to a rank once,
however many of its experts live there).

References independent of the functions under test: a hand-worked fixture, a
cumulative-sum formulation of the per-rank slots, the expert-major layout's
rank counts, the expert-major dispatch's rows for the same tokens, and
round trips that must return x exactly.
"""
import json
import os

import numpy as np
import pytest

import oracle
from combine_moedc_layout_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_rank_layout_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "layout_t4_k2_e4_r2.json")))
    inr = np.array(g["is_token_in_rank"], np.uint8)
    out = oracle.rank_layout(inr, cap_rank=4)
    # rank 0 receives tokens 0, 1, 2; rank 1 receives tokens 0, 3
    np.testing.assert_array_equal(out["rank_slot"], [[0, 0], [1, -1], [2, -1], [-1, 1]])
    assert out["status"] == oracle.OK
    assert oracle.rank_layout(inr, cap_rank=2)["status"] == oracle.ERR_CAPACITY


@pytest.mark.parametrize("name", ["tiny", "low16", "default_ll", "imbalanced_small"])
def test_rank_layout_matches_cumsum_and_counts(name):
    c = synth.make_case("imbalanced", T=512) if name == "imbalanced_small" else synth.make_case(name)
    lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    inr = lay["is_token_in_rank"]
    out = oracle.rank_layout(inr, cap_rank=c.T)
    cum = np.cumsum(inr.astype(np.int64), axis=0) - inr
    ref = np.where(inr == 1, cum, -1)
    np.testing.assert_array_equal(out["rank_slot"], ref)
    np.testing.assert_array_equal((out["rank_slot"] >= 0).sum(axis=0), lay["num_tokens_per_rank"])


@pytest.mark.parametrize("fp8", [False, True])
def test_rank_dispatch_rows_match_tokens_and_expert_dispatch(fp8):
    c = synth.make_case("low16")
    lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    rl = oracle.rank_layout(lay["is_token_in_rank"], cap_rank=c.T)
    rd = oracle.rank_dispatch(c.x, rl["rank_slot"], c.T, fp8=fp8)
    ed = oracle.dispatch(c.x, c.topk_idx, lay["slot"], c.E, c.cap, fp8=fp8)
    epr = c.E // c.R
    for t in range(c.T):
        for r in range(c.R):
            j = rl["rank_slot"][t, r]
            if j < 0:
                continue
            assert rd["rank_src_idx"][r, j] == t
            if not fp8:
                np.testing.assert_array_equal(rd["recv_rank"][r, j], c.x[t])
            # the token's row is the same bytes as its expert-major row for any
            # of its experts on that rank
            k = [k for k in range(c.K) if c.topk_idx[t, k] // epr == r][0]
            e, s = c.topk_idx[t, k], lay["slot"][t, k]
            np.testing.assert_array_equal(rd["recv_rank"][r, j], ed["recv"][e, s])
            if fp8:
                np.testing.assert_array_equal(rd["scales_rank"][r, j], ed["scales"][e, s])
    cnt = lay["num_tokens_per_rank"]
    for r in range(c.R):
        assert (rd["rank_src_idx"][r, cnt[r]:] == -1).all()


def test_rank_combine_round_trips():
    c = synth.make_case("tiny")
    lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    inr = lay["is_token_in_rank"]
    rl = oracle.rank_layout(inr, cap_rank=c.T)
    rd = oracle.rank_dispatch(c.x, rl["rank_slot"], c.T, fp8=False)
    n_ranks = inr.sum(axis=1)
    x = oracle.bf16_to_f32(c.x)
    # every rank returns x / (number of ranks of the token): powers of two make
    # the parts exact, and their sum is x again
    parts = rd["recv_rank"].copy()
    for t in range(c.T):
        if n_ranks[t] in (1, 2, 4):
            for r in np.nonzero(inr[t])[0]:
                parts[r, rl["rank_slot"][t, r]] = synth.f32_to_bf16_bits(
                    x[t] / np.float32(n_ranks[t]))
    y = oracle.rank_combine(parts, rl["rank_slot"])
    sel = np.isin(n_ranks, (1, 2, 4))
    assert sel.sum() > 10
    np.testing.assert_array_equal(y[sel], c.x[sel])
    assert (y[n_ranks == 0] == 0).all()


def test_rank_combine_ascending_order_and_absent_ranks():
    # ranks 0, 1, 2 return 2^24, 1, -2^24: ascending-r binary32 sums give +0
    part = np.array([[[0x4B80]], [[0x3F80]], [[0xCB80]]], np.uint16)
    slot = np.array([[0, 0, 0], [-1, -1, -1]], np.int32)
    y = oracle.rank_combine(part, slot)
    assert y[0, 0] == 0x0000 and y[1, 0] == 0x0000


def test_rank_major_writes_fewer_rows_on_the_4096_token_workload():
    c = synth.make_case("throughput")
    lay = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    rows_rank = int(lay["num_tokens_per_rank"].sum())
    rows_expert = int(lay["num_tokens_per_expert"].sum())
    # 8 experts of 256 over 8 ranks land on ~8 * (1 - (7/8)^8) = 5.25 distinct ranks
    assert abs(rows_rank / c.T - 8 * (1 - (7 / 8) ** 8)) < 0.1
    assert rows_rank < 0.7 * rows_expert
