"""The allocation-free scale entry point.

repro_wscale_noalloc exists for callers that cannot give the library any
device memory -- their allocations belong to another owner, or their loop must
never call cudaMalloc because it would synchronise the device.  Its scratch is
a fixed array inside the library that every call reuses, so these tests call it
through the C ABI several times in a row, on inputs of different sizes, and
require exactly the bits of repro_wscale (which takes a caller workspace).
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

from bitwise_reproducible_int8_gb300 import repro as R  # noqa: E402

REPRO_NOALLOC_MAX_N = 535822336


def _noalloc(x, mode, out):
    return R.lib().repro_wscale_noalloc(
        ctypes.c_void_p(x.data_ptr()), x.numel(), mode, 127, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _bits(t):
    return int(t.view(torch.int32).item())


@pytest.mark.parametrize("mode", [0, 1])
def test_noalloc_matches_the_workspace_entry_point(mode):
    R.repro_set_launch_cfg(reset=True)
    rng = np.random.default_rng(42 + mode)
    # the largest first: the calls after it reuse a scratch array that still
    # holds its partials
    sizes = [23068672, 8192 * 3 + 17, 1000, 1]
    for n in sizes:
        x = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)).cuda()
        ref = torch.empty(1, device="cuda")
        R.repro_wscale(x, mode, ref)
        for _ in range(2):
            out = torch.full((1,), float("nan"), device="cuda")
            assert _noalloc(x, mode, out) == R.REPRO_OK
            torch.cuda.synchronize()
            assert _bits(out) == _bits(ref), (mode, n)
    assert R.repro_device_check() == R.REPRO_OK


def test_noalloc_rejects_sizes_beyond_its_scratch():
    x = torch.zeros(16, device="cuda")
    out = torch.zeros(1, device="cuda")
    st = R.lib().repro_wscale_noalloc(ctypes.c_void_p(x.data_ptr()), REPRO_NOALLOC_MAX_N + 1,
                                      0, 127, ctypes.c_void_p(out.data_ptr()), None)
    assert st == -2                                  # REPRO_ERR_SHAPE, nothing launched
    assert _noalloc(x, 0, out) == R.REPRO_OK        # a valid call right after works
