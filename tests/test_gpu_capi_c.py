"""The plain-C caller (tests/capi/moe_round.c) built and run on the GPU: layout,
dispatch and combine through the C ABI with no Python in the data path; the
program checks its own results (exact K = 1 round trip, slot order, src_idx)."""
import subprocess

import pytest

from test_capi_host import _build_c_caller

pytestmark = pytest.mark.gpu


def test_plain_c_caller_runs(tmp_path):
    from combine_moedc_layout_gb300 import build as mbuild
    mbuild.build()
    exe = _build_c_caller(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "moe_round: ok" in r.stdout
