"""moedc_layout_static_scratch: the layout entry point for callers that cannot
allocate device memory (hosts without a device allocator of their own,
plugins inside a framework whose pool owns the GPU, serving loops that may
not call cudaMalloc once running).  It keeps its scratch in a fixed array
inside the library instead of taking a workspace.

Checked through the C ABI against moedc_layout (which takes a caller-owned
workspace): every output must match exactly (the layout is integer work), on
two calls in a row with different routing, so that leftovers of the first
call cannot leak into the second.  The file is named to run last; it also
passes on its own in a fresh process, where its first call performs the
one-time address lookup.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moedc_layout_gb300 import moedc, synth

pytestmark = pytest.mark.gpu


def _outputs(T, K, E, R):
    dev = "cuda"
    return dict(cnt=torch.full((E,), -7, dtype=torch.int32, device=dev),
                rk=torch.full((R,), -7, dtype=torch.int32, device=dev),
                inr=torch.full((T, R), 9, dtype=torch.uint8, device=dev),
                slot=torch.full((T, K), -7, dtype=torch.int32, device=dev),
                st=torch.zeros(1, dtype=torch.int32, device=dev))


def _reference(idx, T, K, E, R, cap):
    o = _outputs(T, K, E, R)
    ws = moedc.layout_workspace(T, K, E, R, "cuda")
    wsb = 0 if ws is None else ws.numel()
    assert moedc.moedc_layout(idx, T, K, E, R, cap, o["cnt"], o["rk"], o["inr"], o["slot"], ws,
                              wsb, o["st"]) == moedc.OK
    return o


def _static(idx, T, K, E, R, cap):
    o = _outputs(T, K, E, R)
    assert moedc.moedc_layout_static_scratch(idx, T, K, E, R, cap, o["cnt"], o["rk"], o["inr"],
                                             o["slot"], o["st"]) == moedc.OK
    return o


def _same(a, b):
    for key in ("cnt", "rk", "inr", "slot", "st"):
        np.testing.assert_array_equal(a[key].cpu().numpy(), b[key].cpu().numpy(), err_msg=key)


CASES = [
    # more than 65536 (token, k) entries: the layout runs its two-kernel path,
    # which is the one that needs scratch
    lambda: synth.make_random_case(40, T=12000, H=128, K=8, E=256, R=8, cap=None,
                                   dtype=synth.BF16),
    # more tokens, masked entries, different expert / rank counts
    lambda: synth.make_random_case(41, T=40000, H=128, K=8, E=128, R=8, cap=None,
                                   dtype=synth.BF16, mask_p=0.02),
]


def test_static_scratch_matches_workspace_entry_point_twice_in_a_row():
    for make in CASES:                       # two different routings, back to back
        c = make()
        T, K, E, R, cap = c.T, c.K, c.E, c.R, c.cap
        assert 0 < moedc.moedc_layout_workspace_bytes(T, K, E, R) <= moedc.STATIC_SCRATCH_BYTES
        idx = torch.from_numpy(c.topk_idx).cuda()
        ref = _reference(idx, T, K, E, R, cap)
        got = _static(idx, T, K, E, R, cap)
        torch.cuda.synchronize()
        _same(ref, got)
        assert int(got["st"].item()) == 0


def test_static_scratch_second_call_not_polluted_by_first():
    a = synth.make_random_case(42, T=9000, H=128, K=8, E=256, R=8, cap=None, dtype=synth.BF16)
    b = synth.make_random_case(43, T=12000, H=128, K=6, E=64, R=4, cap=None, dtype=synth.BF16,
                               mask_p=0.1)
    for c in (a, b):
        assert moedc.moedc_layout_workspace_bytes(c.T, c.K, c.E, c.R) > 0
    ia = torch.from_numpy(a.topk_idx).cuda()
    ib = torch.from_numpy(b.topk_idx).cuda()
    got_a = _static(ia, a.T, a.K, a.E, a.R, a.cap)
    got_b = _static(ib, b.T, b.K, b.E, b.R, b.cap)
    ref_a = _reference(ia, a.T, a.K, a.E, a.R, a.cap)
    ref_b = _reference(ib, b.T, b.K, b.E, b.R, b.cap)
    torch.cuda.synchronize()
    _same(ref_a, got_a)
    _same(ref_b, got_b)


def test_static_scratch_rejects_shapes_beyond_its_size():
    # 131072 tokens x 8 with 1024 experts and ranks needs 8 MiB of scratch > 1 MiB.
    T, K, E, R = 131072, 8, 1024, 1024
    assert moedc.moedc_layout_workspace_bytes(T, K, E, R) > moedc.STATIC_SCRATCH_BYTES
    # real, full-size buffers, so nothing could go out of bounds even if it launched
    idx = torch.zeros((T, K), dtype=torch.int32, device="cuda")
    o = _outputs(T, K, E, R)
    assert moedc.moedc_layout_static_scratch(idx, T, K, E, R, T * K, o["cnt"], o["rk"], o["inr"],
                                             o["slot"], o["st"]) == moedc.ERR_ARG
    torch.cuda.synchronize()
    assert (o["cnt"].cpu().numpy() == -7).all()      # nothing was launched
    assert int(o["st"].item()) == 0


def _same_as_oracle(got, c):
    ref = oracle.layout(c.topk_idx, c.E, c.R, c.cap)
    np.testing.assert_array_equal(got["cnt"].cpu().numpy(), ref["num_tokens_per_expert"])
    np.testing.assert_array_equal(got["rk"].cpu().numpy(), ref["num_tokens_per_rank"])
    np.testing.assert_array_equal(got["inr"].cpu().numpy(), ref["is_token_in_rank"])
    np.testing.assert_array_equal(got["slot"].cpu().numpy(), ref["slot"])
    assert int(got["st"].item()) == ref["status"]


@pytest.mark.parametrize("shape", [
    # two kernels with scratch (beyond 65536 entries)
    dict(seed=44, T=12000, H=8, K=8, E=256, R=8, cap=None, dtype=synth.BF16, mask_p=0.05),
    # the single-pass layout, its scratch in the static array too (4096 tokens)
    dict(seed=45, T=4096, H=8, K=8, E=256, R=8, cap=None, dtype=synth.BF16),
    # the sweep (1024 entries): no scratch, so no address lookup
    dict(seed=47, T=128, H=8, K=8, E=288, R=8, cap=None, dtype=synth.BF16, mask_p=0.05),
    # K = 6: 4 chunks of floor(1024 / 6) tokens at 511 tokens (3066 entries), the single pass
    dict(seed=48, T=511, H=8, K=6, E=60, R=6, cap=None, dtype=synth.BF16),
])
def test_static_scratch_matches_oracle_directly(shape):
    c = synth.make_random_case(**shape)
    idx = torch.from_numpy(c.topk_idx).cuda()
    for _ in range(2):                      # twice in a row on the shared array
        got = _static(idx, c.T, c.K, c.E, c.R, c.cap)
        torch.cuda.synchronize()
        _same_as_oracle(got, c)


def test_static_scratch_call_allocates_nothing():
    """After a first call on the device (which looks up the array's address),
    further calls change neither torch's allocator nor the device's free
    memory: the scratch is the array inside the library."""
    c = synth.make_random_case(46, T=12000, H=8, K=8, E=256, R=8, cap=None, dtype=synth.BF16)
    idx = torch.from_numpy(c.topk_idx).cuda()
    o = _outputs(c.T, c.K, c.E, c.R)

    def call():
        assert moedc.moedc_layout_static_scratch(idx, c.T, c.K, c.E, c.R, c.cap, o["cnt"],
                                                 o["rk"], o["inr"], o["slot"],
                                                 o["st"]) == moedc.OK

    call()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    _same_as_oracle(o, c)
