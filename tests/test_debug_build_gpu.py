"""The -DWAN_DEBUG library on the GPU: the parity tests pass under it with
every device-side invariant check live, and a forced check failure comes back
as WAN_ERR_DEVICE_CHECK with its source line, leaving the context usable.

Each run is a subprocess whose binding loads the debug library (WAN_ATTN_LIB),
so that this process keeps the release library.
"""
import os
import subprocess
import sys

import pytest

from long_sequence_attention_02_b300 import build

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _env():
    env = dict(os.environ)
    env["WAN_ATTN_LIB"] = build.build_attn(debug=True)
    return env


def test_parity_tests_pass_under_the_debug_library():
    tests = ["tests/test_fwd_gpu.py", "tests/test_bwd_gpu.py", "tests/test_fp8_gpu.py",
             "tests/test_conv3d_gpu.py", "tests/test_time_down_gpu.py", "tests/test_ring_dual_gpu.py"]
    sel = "every_row or every_output or exhaustive or chunks or first_chunk"
    r = subprocess.run([sys.executable, "-m", "pytest", *tests, "-m", "gpu", "-q", "-x", "-k", sel,
                        "-p", "no:cacheprovider"], cwd=ROOT, env=_env(), capture_output=True, text=True,
                       timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " deselected" in r.stdout


CHECK_SCRIPT = r"""
import math, torch
import long_sequence_attention_02_b300 as wan
assert wan.wan_debug_build() == 1, "not the debug library"
grid, B, H = (3, 8, 8), 1, 2
L = grid[0] * grid[1] * grid[2]
q = torch.randn(B, L, H, 128, device="cuda").bfloat16()
k, v = torch.randn_like(q), torch.randn_like(q)
o1, _ = wan.attention_forward(q, k, v, grid)
assert wan.wan_get_device_status() == wan.WAN_OK
wan.check(wan.wan_debug_inject_check(1))
o2, _ = wan.attention_forward(q, k, v, grid)          # entry check fails; the work still runs
st = wan.wan_get_device_status()
line = wan.wan_debug_check_line()
o3, _ = wan.attention_forward(q, k, v, grid)
st2 = wan.wan_get_device_status()
print("status", st, "line", line, "after", st2)
assert st == wan.WAN_ERR_DEVICE_CHECK and line > 0 and st2 == wan.WAN_OK
assert torch.equal(o1, o2) and torch.equal(o1, o3)
"""


def test_forced_check_is_reported_with_its_line():
    r = subprocess.run([sys.executable, "-c", CHECK_SCRIPT], cwd=ROOT, env=_env(), capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
