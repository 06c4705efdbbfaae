"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every entry point the header declares, and rejects bad
arguments before touching CUDA.  Also the benchmark's byte accounting and
its multi-rank reduction (gloo, two processes)."""
import ctypes
import os
import re
import subprocess

import pytest

from combine_moedc_layout_gb300 import build as mbuild
from combine_moedc_layout_gb300 import moedc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return moedc.load()


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"MOEDC_EXPORT\s+[\w\s\*]+?\b(moedc_\w+)\s*\(", src))
    return names


def test_header_declares_expected_entry_points():
    names = declared_symbols()
    assert {"moedc_layout", "moedc_dispatch", "moedc_combine", "moedc_layout_dispatch",
            "moedc_strerror", "moedc_api_version", "moedc_layout_workspace_bytes"} <= names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", mbuild.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(moedc_\w+)", out))
    missing = declared_symbols() - exported
    assert not missing, missing
    for name in declared_symbols():
        assert hasattr(lib, name)
    # nothing but the declared C entry points is visible
    assert exported == declared_symbols()


def test_version_and_strerror(lib):
    assert lib.moedc_api_version() == 1
    for code in range(7):
        assert moedc.strerror(code) and "unknown" not in moedc.strerror(code)
    assert "unknown" in moedc.strerror(99)


def _onepass_bytes(T, K, E, R):
    """Single-pass layout workspace: a 256-byte header (the generation word),
    then one row of E + R tagged 64-bit counts per chunk, then two spare
    words.  A chunk holds 1024 * ept // K tokens with the smallest ept in
    (1, 2, 4) that keeps it to at most 144 chunks; 0 below 4 chunks of 1024
    entries (the sweep runs) and beyond 144 chunks at ept 4."""
    for ept in (1, 2, 4):
        chunks = max(1, -(-T // (1024 * ept // K)))
        if ept == 1 and chunks < 4:
            return 0
        if chunks <= 144:
            return 256 + (chunks * (E + R) + 2) * 8
    return 0


def _blocked_bytes(T, K, E, R):
    """The two-kernel layout's counts beyond 65536 entries: blocks of
    max(ceil(1024 / K), ceil(T / 1024)) tokens, (E + R) int32 each."""
    if T * K <= 65536:
        return 0
    tpc = max(-(-1024 // K), -(-T // 1024))
    return -(-T // tpc) * (E + R) * 4


def test_workspace_bytes(lib):
    # up to 3072 entries (fewer than 4 chunks): the sweep, no workspace
    assert moedc.moedc_layout_workspace_bytes(64, 4, 32, 4) == 0
    assert moedc.moedc_layout_workspace_bytes(128, 8, 288, 8) == 0
    assert moedc.moedc_layout_workspace_bytes(384, 8, 256, 8) == 0
    assert moedc.moedc_layout_workspace_bytes(0, 8, 256, 8) == 0
    # a chunk holds floor(1024 / K) tokens, so where K does not divide 1024
    # the single pass starts a little below 3072 entries
    for T, K, first in [(510, 6, False), (511, 6, True), (1023, 3, False), (1024, 3, True),
                        (612, 5, False), (613, 5, True), (438, 7, False), (439, 7, True)]:
        got = moedc.moedc_layout_workspace_bytes(T, K, 42, 6)
        assert got == _onepass_bytes(T, K, 42, 6), (T, K)
        assert (got > 0) == first, (T, K, got)
    # from 4 chunks to 65536 entries: the single-pass layout's (optional) workspace
    assert moedc.moedc_layout_workspace_bytes(512, 8, 256, 8) == _onepass_bytes(512, 8, 256, 8) > 0
    assert moedc.moedc_layout_workspace_bytes(4096, 8, 256, 8) == 256 + (32 * 264 + 2) * 8
    assert moedc.moedc_layout_workspace_bytes(8192, 8, 256, 8) == _onepass_bytes(8192, 8, 256, 8)
    assert moedc.moedc_layout_workspace_bytes(2048, 32, 1024, 1024) == \
        _onepass_bytes(2048, 32, 1024, 1024)
    # beyond 65536 entries: the larger of the single-pass rows and the
    # two-kernel layout's counts (blocks x (E + R) int32)
    assert _blocked_bytes(8193, 8, 256, 8) == 65 * (256 + 8) * 4
    assert _onepass_bytes(8193, 8, 256, 8) == 256 + (65 * 264 + 2) * 8
    assert moedc.moedc_layout_workspace_bytes(8193, 8, 256, 8) == 256 + (65 * 264 + 2) * 8
    assert _blocked_bytes(40000, 8, 128, 8) == 313 * (128 + 8) * 4
    assert _onepass_bytes(40000, 8, 128, 8) == 256 + (79 * 136 + 2) * 8     # 4 per thread
    assert moedc.moedc_layout_workspace_bytes(40000, 8, 128, 8) == 313 * (128 + 8) * 4
    assert _onepass_bytes(20000, 8, 128, 8) == 256 + (79 * 136 + 2) * 8     # 2 per thread
    for shape in [(12000, 8, 256, 8), (20000, 8, 128, 8), (90000, 6, 60, 6), (120000, 6, 60, 6),
                  (16384, 8, 1024, 1024)]:
        assert moedc.moedc_layout_workspace_bytes(*shape) == max(_onepass_bytes(*shape),
                                                                 _blocked_bytes(*shape)), shape
    assert _onepass_bytes(120000, 6, 60, 6) == 0          # beyond 144 chunks of 4096 entries
    # the one-call layout+dispatch: the layout's workspace while the layout
    # is one launch (fused block, or layout then dispatch), beyond it the
    # cooperative launch's barrier words and count rows [E + R][2048]
    assert moedc.moedc_layout_dispatch_workspace_bytes(128, 8, 288, 8) == 0
    assert moedc.moedc_layout_dispatch_workspace_bytes(4096, 8, 256, 8) == \
        _onepass_bytes(4096, 8, 256, 8)
    assert moedc.moedc_layout_dispatch_workspace_bytes(8193, 8, 256, 8) == 256 + 264 * 2048 * 4
    assert moedc.moedc_layout_dispatch_workspace_bytes(40000, 8, 128, 8) == 256 + 136 * 2048 * 4
    assert moedc.moedc_layout_dispatch_workspace_bytes(4096, 8, 250, 8) == 0
    # rejected shapes report 0
    assert moedc.moedc_layout_workspace_bytes(4096, 8, 250, 8) == 0
    assert moedc.moedc_layout_workspace_bytes(4096, 0, 256, 8) == 0


def test_argument_errors_return_before_cuda(lib):
    P = ctypes.c_void_p
    fake = P(256)             # never dereferenced: validation fails first
    # K = 0, E % R != 0, E too large, cap = 0
    for (T, K, E, R, cap) in [(4, 0, 8, 2, 4), (4, 2, 9, 2, 4), (4, 2, 2048, 2, 4),
                              (4, 2, 8, 2, 0), (-1, 2, 8, 2, 4), (4, 33, 64, 2, 4)]:
        assert lib.moedc_layout(fake, T, K, E, R, cap, fake, fake, fake, fake, None, 0, fake,
                                None) == moedc.ERR_ARG
    # dispatch: fp8 with H % 128 != 0; bad dtype; null scales for fp8
    assert lib.moedc_dispatch(fake, 4, 200, fake, fake, fake, 2, 8, 4, moedc.FP8_E4M3, fake,
                              fake, fake, fake, None) == moedc.ERR_ARG
    assert lib.moedc_dispatch(fake, 4, 256, fake, fake, fake, 2, 8, 4, 7, fake, fake, fake,
                              fake, None) == moedc.ERR_ARG
    assert lib.moedc_dispatch(fake, 4, 256, fake, fake, fake, 2, 8, 4, moedc.FP8_E4M3, fake,
                              None, fake, fake, None) == moedc.ERR_ARG
    # misaligned x (bf16 needs 16-byte alignment)
    assert lib.moedc_dispatch(P(258), 4, 256, fake, fake, fake, 2, 8, 4, moedc.BF16, fake,
                              None, fake, fake, None) == moedc.ERR_ARG
    # combine: H % 8 != 0, null y
    assert lib.moedc_combine(fake, 8, 4, 100, fake, fake, fake, 4, 2, fake, fake, None) == \
        moedc.ERR_ARG
    assert lib.moedc_combine(fake, 8, 4, 128, fake, fake, fake, 4, 2, None, fake, None) == \
        moedc.ERR_ARG
    # e4m3 combine / dequant: unknown scale layout, H % 128 != 0; dispatch: unknown dtype bits
    assert lib.moedc_combine_e4m3(fake, fake, 7, 8, 4, 256, fake, fake, fake, 4, 2, fake, fake,
                                  None) == moedc.ERR_ARG
    assert lib.moedc_combine_e4m3(fake, fake, 0, 8, 4, 200, fake, fake, fake, 4, 2, fake, fake,
                                  None) == moedc.ERR_ARG
    assert lib.moedc_dequant_e4m3(fake, fake, 3, fake, 8, 4, 256, fake, None) == moedc.ERR_ARG
    # per-token scales: not with the column-major flag, not beyond the width limit, not on
    # the rank-major path, not as a bf16 flag
    both = moedc.FP8_E4M3 | moedc.SCALES_PER_TOKEN | moedc.SCALES_COL_MAJOR
    assert lib.moedc_dispatch(fake, 4, 256, fake, fake, fake, 2, 8, 4, both, fake, fake, fake,
                              fake, None) == moedc.ERR_ARG
    tok = moedc.FP8_E4M3 | moedc.SCALES_PER_TOKEN
    wide = moedc.TOKEN_SCALE_MAX_H + 128
    assert lib.moedc_dispatch(fake, 4, wide, fake, fake, fake, 2, 8, 4, tok, fake, fake, fake,
                              fake, None) == moedc.ERR_ARG
    assert lib.moedc_layout_dispatch(fake, fake, 4, wide, 2, 8, 2, 4, tok, fake, fake, fake,
                                     fake, fake, fake, fake, None, 0, fake, None) == moedc.ERR_ARG
    assert lib.moedc_dispatch(fake, 4, 256, fake, fake, fake, 2, 8, 4,
                              moedc.BF16 | moedc.SCALES_PER_TOKEN, fake, fake, fake, fake,
                              None) == moedc.ERR_ARG
    assert lib.moedc_rank_dispatch(fake, 4, 256, fake, fake, 2, 4, tok, fake, fake, fake,
                                   None) == moedc.ERR_ARG
    assert lib.moedc_combine_e4m3(fake, fake, moedc.SCALES_PER_TOKEN | moedc.SCALES_COL_MAJOR, 8,
                                  4, 256, fake, fake, fake, 4, 2, fake, fake, None) == \
        moedc.ERR_ARG
    assert lib.moedc_dispatch(fake, 4, 256, fake, fake, fake, 2, 8, 4,
                              moedc.BF16 | moedc.SCALES_COL_MAJOR, fake, fake, fake, fake,
                              None) == moedc.ERR_ARG
    # fused: a shape past the single-launch layout (> 65536 entries) without workspace
    assert lib.moedc_layout_dispatch(fake, fake, 9000, 256, 8, 64, 8, 1200, moedc.BF16, fake,
                                     fake, fake, fake, fake, None, fake, None, 0, fake,
                                     None) == moedc.ERR_ARG


def test_bench_byte_accounting():
    import bench
    b = bench.algorithmic_bytes(T=4096, H=7168, K=8, E=256, R=8, cap=160, N=32768, fp8=True)
    # read x once per token + 32768 e4m3 rows with 56 fp32 scales + idx/slot + src_idx
    assert b["dispatch"] == 2 * 7168 * 4096 + 32768 * (7168 + 224) + 8 * 4096 * 8 + 4 * 256 * 160
    assert abs(b["dispatch"] / 1e6 - 301.4) < 0.1
    assert abs(b["combine"] / 1e6 - 528.9) < 0.1
    assert bench.whole_job_gbs(10**9, 2, 1.0) == pytest.approx(2000.0)


def _gloo_worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(1.0 + rank, world)
    q.put((rank, slowest, bench.whole_job_gbs(10**9, world, slowest)))
    dist.destroy_process_group()


def test_bench_max_over_ranks_gloo_two_processes():
    import multiprocessing as mp
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_gloo_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [2.0, 2.0]            # both see the slowest rank
    assert all(abs(r[2] - 1000.0) < 1e-9 for r in res)  # 2 x 1 GB / 2 ms


def test_missing_library_fails_loudly(tmp_path):
    """No CPU fallback: without the built library every call raises."""
    with pytest.raises(RuntimeError, match="not found"):
        moedc.load(str(tmp_path / "libmoedc.so"))


def test_product_package_does_not_import_the_oracle():
    import combine_moedc_layout_gb300 as pkg
    pkg_dir = os.path.dirname(pkg.__file__)
    for root, _, files in os.walk(pkg_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(root, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "moedc_oracle" not in src, f


def _build_c_caller(tmp_path):
    """Compile tests/capi/moe_round.c as C11 against include/moedc.h and link it
    to libmoedc.so and the CUDA runtime; returns the executable's path."""
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "moe_round")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "capi", "moe_round.c"), "-o", exe,
           "-L" + os.path.dirname(mbuild.LIB_PATH), "-lmoedc",
           "-L" + os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.dirname(mbuild.LIB_PATH)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_plain_c_caller_compiles_and_links(lib, tmp_path):
    """The header is valid C11 and a C program links against the library
    with no C++ or Python in between (running it needs a GPU: see
    test_gpu_capi_c.py)."""
    assert os.path.exists(_build_c_caller(tmp_path))


def test_bench_threaded_oracle_step_matches_single_thread():
    """The all-cores CPU baseline splits dispatch and combine by token runs over
    threads; its outputs must equal the single-threaded oracle step bit for
    bit (the bench asserts the same on the full workload)."""
    from concurrent.futures import ThreadPoolExecutor

    import bench
    from combine_moedc_layout_gb300 import synth
    c = synth.make_case("throughput")
    c.extra["eo_host"] = synth.make_expert_out(c, 0)
    assert bench._token_chunks(10, 4) == [(0, 2), (2, 5), (5, 7), (7, 10)]
    assert bench._token_chunks(3, 8) == [(0, 1), (1, 2), (2, 3)]
    _, b1, one = bench.oracle_step(c, 96, keep=True)
    with ThreadPoolExecutor(max_workers=4) as pool:
        _, b4, four = bench.oracle_step(c, 96, threads=4, pool=pool, keep=True)
    assert b1 == b4
    assert bench.same_oracle_outputs(one, four)
    four["y"][0, 0] ^= 1                       # a planted difference is caught
    assert not bench.same_oracle_outputs(one, four)


def test_bench_arms_share_one_config_and_report_the_cpu():
    import bench
    from combine_moedc_layout_gb300 import synth
    c = synth.make_case("throughput")
    a, b = bench.workload_config(c, 1), bench.workload_config(c, 1)
    assert a == b and {"workload", "T", "H", "K", "E", "R", "cap", "parallelism", "l2"} <= set(a)
    assert bench.host_cores() >= 1
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
