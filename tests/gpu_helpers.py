"""Helpers for the GPU parity tests: move numpy arrays to cuda:0, run the
library's calls, compare bit patterns with the oracle's."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import bitwise_reproducible_int8_gb300 as R  # noqa: E402


def dev(a) -> "torch.Tensor":
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def host(t) -> np.ndarray:
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def scalar(v) -> "torch.Tensor":
    return torch.tensor([float(v)], dtype=torch.float32, device="cuda")


def assert_bits_equal(got, exp, what=""):
    got = np.ascontiguousarray(got)
    exp = np.ascontiguousarray(exp)
    assert got.shape == exp.shape, (what, got.shape, exp.shape)
    if got.dtype == np.float32:
        g, e = got.view(np.uint32).ravel(), exp.view(np.uint32).ravel()
    else:
        g, e = got.ravel(), exp.ravel()
    bad = np.flatnonzero(g != e)
    if bad.size:
        i = bad[0]
        msg = f"{what}: {bad.size} of {g.size} differ; first at flat index {i}: " \
              f"got {got.ravel()[i]!r} (0x{int(g[i]) & 0xffffffff:08x}) " \
              f"expected {exp.ravel()[i]!r} (0x{int(e[i]) & 0xffffffff:08x})"
        if got.dtype == np.float32:
            ulp = abs(int(g[i].astype(np.int64)) - int(e[i].astype(np.int64)))
            msg += f", {ulp} ulp"
        raise AssertionError(msg)


def gpu_scale(x: np.ndarray, mode: int) -> np.float32:
    xt = dev(x.ravel())
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    R.repro_wscale(xt, mode, s)
    return host(s)[0]


def gpu_quant(x: np.ndarray, s: float) -> np.ndarray:
    xt = dev(x)
    q = torch.empty(x.shape, dtype=torch.int8, device="cuda")
    R.repro_quant_i8(xt, scalar(s), q)
    return host(q)


def gpu_fwd(xq, wq, s_x, s_w) -> np.ndarray:
    M, N = xq.shape[0], wq.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    R.repro_linear_fwd(dev(xq), dev(wq), scalar(s_x), scalar(s_w), y)
    return host(y)


def gpu_bwd(dy, xq, wq, s_x, s_w, want_dx=True, want_dw=True):
    M, N = dy.shape
    K = (xq if xq is not None else wq).shape[1]
    dx = torch.empty((M, K), dtype=torch.float32, device="cuda") if want_dx else None
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda") if want_dw else None
    R.repro_linear_bwd(dev(dy), dev(xq) if xq is not None else None,
                       dev(wq) if wq is not None else None,
                       scalar(s_x) if s_x is not None else None,
                       scalar(s_w) if s_w is not None else None, dx, dw)
    return (host(dx) if want_dx else None), (host(dw) if want_dw else None)


def gpu_treefold(parts) -> np.ndarray:
    ts = [dev(p) for p in parts]
    out = torch.empty_like(ts[0])
    R.repro_treefold(ts, out)
    return host(out)


def gpu_accum(acc, g) -> np.ndarray:
    a = dev(acc.copy())
    R.repro_grad_accum(a, dev(g))
    return host(a)
