"""The allocation-free scale entry point.

repro_wscale_noalloc exists for callers that cannot give the library any
device memory -- their allocations belong to another owner, or their loop must
never call cudaMalloc because it would synchronise the device.  Its scratch is
a fixed array inside the library that every call reuses, so these tests call it
through the C ABI several times in a row, on inputs of different sizes, and
require exactly the bits of the CPU oracle and of repro_wscale (which takes a
caller workspace), up to the largest size the header accepts.
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
def test_noalloc_matches_the_workspace_entry_point(orc, mode):
    R.repro_set_launch_cfg(reset=True)
    rng = np.random.default_rng(42 + mode)
    # the largest first: the calls after it reuse a scratch array that still
    # holds its partials
    sizes = [23068672, 8192 * 3 + 17, 1000, 1]
    for n in sizes:
        xh = (rng.standard_normal(n) * 0.02).astype(np.float32)
        x = torch.from_numpy(xh).cuda()
        ref = torch.empty(1, device="cuda")
        R.repro_wscale(x, mode, ref)
        exp = int(np.float32(orc.wscale(xh, mode)).view(np.int32))
        assert _bits(ref) == exp, (mode, n)
        for _ in range(2):
            out = torch.full((1,), float("nan"), device="cuda")
            assert _noalloc(x, mode, out) == R.REPRO_OK
            torch.cuda.synchronize()
            assert _bits(out) == exp, (mode, n)
    assert R.repro_device_check() == R.REPRO_OK


def test_noalloc_at_the_largest_accepted_size(orc):
    # n = REPRO_NOALLOC_MAX_N fills the scratch array exactly with the weight
    # scale's partials (65408 block sums, then the tree pass's and the slack);
    # 2.1 GB of fp32 on the device
    n = REPRO_NOALLOC_MAX_N
    xh = np.empty(n, dtype=np.float32)
    step = 1 << 24
    for lo in range(0, n, step):   # a fixed mixed-sign pattern, built in slices
        i = np.arange(lo, min(lo + step, n), dtype=np.int64)
        xh[lo:lo + i.size] = (i * 7919 % 2001 - 1000).astype(np.float32) * np.float32(1e-5)
    x = torch.from_numpy(xh).cuda()
    for mode in (0, 1):
        exp = int(np.float32(orc.wscale(xh, mode)).view(np.int32))
        ref = torch.empty(1, device="cuda")
        R.repro_wscale(x, mode, ref)
        for _ in range(2):
            out = torch.full((1,), float("nan"), device="cuda")
            assert _noalloc(x, mode, out) == R.REPRO_OK
            torch.cuda.synchronize()
            assert _bits(out) == exp, mode
        assert _bits(ref) == exp, mode
    del x
    torch.cuda.empty_cache()
    assert R.repro_device_check() == R.REPRO_OK


def test_noalloc_rejects_sizes_beyond_its_scratch():
    x = torch.zeros(16, device="cuda")
    out = torch.zeros(1, device="cuda")
    st = R.lib().repro_wscale_noalloc(ctypes.c_void_p(x.data_ptr()), REPRO_NOALLOC_MAX_N + 1,
                                      0, 127, ctypes.c_void_p(out.data_ptr()), None)
    assert st == -2                                  # REPRO_ERR_SHAPE, nothing launched
    assert _noalloc(x, 0, out) == R.REPRO_OK        # a valid call right after works
