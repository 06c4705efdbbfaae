"""The GPU's binary32 -> e4m3fn conversion against the oracle's encoder over
every binary32 bit pattern.

The library quantises each binary32 quotient x / s with one hardware
conversion (cvt.rn.satfinite.e4m3x2.f32, round to nearest even, magnitudes
beyond 448 saturated to +-448).  The parity tests reach that instruction only
through the quotients their inputs produce; this test applies the library's
own conversion helper to all 2^32 bit patterns and compares each code with the
oracle's encoder (nearest e4m3fn value by its definition, ties to even,
satfinite), which the CPU tests pin to a brute-force nearest search.  NaN
patterns are left out: the method's inputs are finite.  The sweep kernel lives
in tests/cuda and is built by this test, not into libmoedc.
"""
import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CHUNK = 1 << 26


def _build(tmp_path) -> ctypes.CDLL:
    src = os.path.join(HERE, "cuda", "e4m3_cvt_sweep.cu")
    so = str(tmp_path / "libe4m3_cvt_sweep.so")
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
           "-I" + os.path.join(ROOT, "include"),
           "-I" + os.path.join(ROOT, "combine_moedc_layout_gb300", "csrc"), src, "-o", so]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    lib.e4m3_cvt_sweep.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p,
                                   ctypes.c_void_p]
    lib.e4m3_cvt_sweep.restype = ctypes.c_int
    return lib


def _oracle_codes(f: np.ndarray, pool, parts: int) -> np.ndarray:
    bounds = [len(f) * j // parts for j in range(parts + 1)]
    out = list(pool.map(lambda j: oracle.e4m3_encode(f[bounds[j]:bounds[j + 1]]), range(parts)))
    return np.concatenate(out)


def test_hardware_e4m3_conversion_matches_oracle_on_every_binary32(tmp_path):
    lib = _build(tmp_path)
    out = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    threads = max(1, len(os.sched_getaffinity(0)))
    compared = 0
    nan_patterns = 0
    with ThreadPoolExecutor(max_workers=threads) as pool:
        for base in range(0, 1 << 32, CHUNK):
            assert lib.e4m3_cvt_sweep(base, CHUNK, ctypes.c_void_p(out.data_ptr()),
                                      ctypes.c_void_p(stream.cuda_stream)) == 0
            gpu = out.cpu().numpy()
            bits = np.arange(base, base + CHUNK, dtype=np.uint64).astype(np.uint32)
            ref = _oracle_codes(bits.view(np.float32), pool, threads)
            nan = ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x007FFFFF) != 0)
            bad = (gpu != ref) & ~nan
            if bad.any():
                i = int(np.flatnonzero(bad)[0])
                pytest.fail(f"{int(bad.sum())} codes differ in chunk {base:#x}; first: bits "
                            f"{int(bits[i]):#010x} gpu {int(gpu[i]):#04x} oracle {int(ref[i]):#04x}")
            compared += int((~nan).sum())
            nan_patterns += int(nan.sum())
    # every pattern except the 2 * (2^23 - 1) NaNs was compared
    assert nan_patterns == 2 * ((1 << 23) - 1)
    assert compared == (1 << 32) - nan_patterns
    print(f"e4m3 conversion: {compared} binary32 patterns compared, all equal")
