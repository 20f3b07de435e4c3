"""CPU oracle of the bitwise-reproducible int8 QAT linear layer.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (``bench.py``) may import this package.  The CUDA
library and its Python binding never import it; there is no CPU fallback.

The arithmetic lives in ``oracle.c`` (plain C11, contraction off, subnormals
flushed in software); this module only compiles it and marshals numpy arrays
through ctypes.  See ``oracle.h`` for the definitions and their sources.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

CFLAGS = [
    "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
    "-fexcess-precision=standard", "-fPIC", "-shared",
]


def build(force: bool = False, openmp: bool = True) -> str:
    """Compile oracle.c into liboracle.so next to it; return the path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(os.path.join(_HERE, "oracle.h")))):
        return _LIB_PATH
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found to build the oracle")
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    flags = CFLAGS + (["-fopenmp"] if openmp else [])
    cmd = [cc, *flags, _SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and openmp:
        os.unlink(tmp)
        return build(force=True, openmp=False)
    if r.returncode != 0:
        os.unlink(tmp)
        raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


class AdamWHparams(ctypes.Structure):
    _fields_ = [(k, ctypes.c_float) for k in
                ("lr", "beta1", "beta2", "eps", "weight_decay", "max_norm")]


_f32p = ctypes.POINTER(ctypes.c_float)
_i8p = ctypes.POINTER(ctypes.c_int8)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def load(path: str) -> ctypes.CDLL:
    """Open a compiled oracle library at `path` and declare its signatures
    (the tests also load copies built with a planted mistake)."""
    L = ctypes.CDLL(path)
    sig = {
        "oracle_flush": (ctypes.c_float, [ctypes.c_float]),
        "oracle_add": (ctypes.c_float, [ctypes.c_float, ctypes.c_float]),
        "oracle_mul": (ctypes.c_float, [ctypes.c_float, ctypes.c_float]),
        "oracle_div": (ctypes.c_float, [ctypes.c_float, ctypes.c_float]),
        "oracle_sqrt": (ctypes.c_float, [ctypes.c_float]),
        "oracle_i2f": (ctypes.c_float, [_i64]),
        "oracle_quant_one": (ctypes.c_int, [ctypes.c_float, ctypes.c_float, ctypes.c_int]),
        "oracle_canon_sum": (ctypes.c_float, [_f32p, _i64]),
        "oracle_wscale": (ctypes.c_float, [_f32p, _i64, ctypes.c_int, ctypes.c_int]),
        "oracle_quant_i8": (None, [_f32p, _i64, ctypes.c_float, ctypes.c_int, _i8p]),
        "oracle_linear_fwd": (None, [_i8p, _i8p, ctypes.c_float, ctypes.c_float, _f32p,
                                     _i64, _i64, _i64]),
        "oracle_linear_fwd_at": (None, [_i8p, _i8p, ctypes.c_float, ctypes.c_float,
                                        _i64, _i64, _i64, _i64p, _i64p, _i64, _f32p]),
        "oracle_int_dot": (ctypes.c_int64, [_i8p, _i8p, _i64, _i64, _i64]),
        "oracle_linear_bwd_dx": (None, [_f32p, _i8p, ctypes.c_float, _f32p, _i64, _i64, _i64]),
        "oracle_linear_bwd_dw": (None, [_f32p, _i8p, ctypes.c_float, _f32p, _i64, _i64, _i64]),
        "oracle_linear_bwd_dx_at": (None, [_f32p, _i8p, ctypes.c_float, _i64, _i64, _i64,
                                           _i64p, _i64p, _i64, _f32p]),
        "oracle_linear_bwd_dw_at": (None, [_f32p, _i8p, ctypes.c_float, _i64, _i64, _i64,
                                           _i64p, _i64p, _i64, _f32p]),
        "oracle_grad_accum": (None, [_f32p, _f32p, _i64]),
        "oracle_running_sum": (None, [ctypes.POINTER(_f32p), ctypes.c_int, _i64, _f32p]),
        "oracle_treefold_one": (ctypes.c_float, [_f32p, ctypes.c_int]),
        "oracle_treefold": (None, [ctypes.POINTER(_f32p), ctypes.c_int, _i64, _f32p]),
        "oracle_treefold_all_ranks": (None, [_f32p, ctypes.c_int, _f32p]),
        "oracle_threads": (ctypes.c_int, []),
        "oracle_set_threads": (None, [ctypes.c_int]),
        "oracle_sumsq": (ctypes.c_float, [_f32p, _i64]),
        "oracle_pow_t": (ctypes.c_float, [ctypes.c_float, _i64]),
        "oracle_clip_coef": (ctypes.c_float, [ctypes.c_float, ctypes.c_float]),
        "oracle_adamw_step": (None, [_f32p, _f32p, _f32p, _f32p, _i64, ctypes.c_float,
                                     ctypes.POINTER(AdamWHparams), _i64]),
        "oracle_exp": (ctypes.c_float, [ctypes.c_float]),
        "oracle_attn_quant_p": (ctypes.c_int, [ctypes.c_float]),
        "oracle_attn_fx": (ctypes.c_int64, [ctypes.c_float]),
        "oracle_attn_fix2f": (ctypes.c_float, [_i64]),
        "oracle_attn_fwd": (None, [_f32p, _f32p, _i8p, ctypes.c_float, _f32p, _f32p, _f32p,
                                   _i64, _i64, _i64, _i64, _i64, _i64]),
        "oracle_attn_fwd_rows": (None, [_f32p, _f32p, _i8p, ctypes.c_float, _i64p, _i64,
                                        _f32p, _f32p, _f32p, _i64, _i64, _i64, _i64, _i64,
                                        _i64]),
        "oracle_attn_bwd": (None, [_f32p, _f32p, _i8p, ctypes.c_float, _f32p, _f32p, _f32p,
                                   _f32p, _f32p, _f32p, _f32p, _i64, _i64, _i64, _i64, _i64,
                                   _i64]),
        "oracle_attn_bwd_rows": (None, [_f32p, _f32p, _i8p, ctypes.c_float, _f32p, _f32p,
                                        _f32p, _f32p, _i64p, _i64, _f32p, _i64p, _i64, _f32p,
                                        _f32p, _i64, _i64, _i64, _i64, _i64, _i64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


# ---------------------------------------------------------------- helpers

def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _i8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int8)


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def f32_bits(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).view(np.uint32)


# ---------------------------------------------------------------- elementary ops

def flush(a: float) -> float:
    return lib().oracle_flush(a)


def add(a: float, b: float) -> float:
    return lib().oracle_add(a, b)


def mul(a: float, b: float) -> float:
    return lib().oracle_mul(a, b)


def div(a: float, b: float) -> float:
    return lib().oracle_div(a, b)


def sqrt(a: float) -> float:
    return lib().oracle_sqrt(a)


def i2f(v: int) -> float:
    return lib().oracle_i2f(int(v))


def quant_one(x: float, s: float, qmax: int = 127) -> int:
    return lib().oracle_quant_one(x, s, qmax)


# ---------------------------------------------------------------- the path

def canon_sum(p) -> np.float32:
    p = _f32(p).ravel()
    return np.float32(lib().oracle_canon_sum(_p(p, _f32p), p.size))


def wscale(x, mode: int, qmax: int = 127) -> np.float32:
    x = _f32(x).ravel()
    return np.float32(lib().oracle_wscale(_p(x, _f32p), x.size, int(mode), int(qmax)))


def quant_i8(x, s: float, qmax: int = 127) -> np.ndarray:
    x = _f32(x)
    q = np.empty(x.shape, dtype=np.int8)
    lib().oracle_quant_i8(_p(x, _f32p), x.size, float(s), int(qmax), _p(q, _i8p))
    return q


def linear_fwd(xq, wq, s_x: float, s_w: float) -> np.ndarray:
    xq, wq = _i8(xq), _i8(wq)
    M, K = xq.shape
    N, K2 = wq.shape
    assert K == K2
    y = np.empty((M, N), dtype=np.float32)
    lib().oracle_linear_fwd(_p(xq, _i8p), _p(wq, _i8p), float(s_x), float(s_w),
                            _p(y, _f32p), M, N, K)
    return y


def linear_fwd_at(xq, wq, s_x, s_w, idx_m, idx_n) -> np.ndarray:
    xq, wq = _i8(xq), _i8(wq)
    M, K = xq.shape
    N = wq.shape[0]
    im = np.ascontiguousarray(idx_m, dtype=np.int64)
    jn = np.ascontiguousarray(idx_n, dtype=np.int64)
    out = np.empty(im.size, dtype=np.float32)
    lib().oracle_linear_fwd_at(_p(xq, _i8p), _p(wq, _i8p), float(s_x), float(s_w), M, N, K,
                               _p(im, _i64p), _p(jn, _i64p), im.size, _p(out, _f32p))
    return out


def int_dot(xq, wq, m: int, n: int) -> int:
    xq, wq = _i8(xq), _i8(wq)
    return int(lib().oracle_int_dot(_p(xq, _i8p), _p(wq, _i8p), m, n, xq.shape[1]))


def linear_bwd_dx(dy, wq, s_w: float) -> np.ndarray:
    dy, wq = _f32(dy), _i8(wq)
    M, N = dy.shape
    N2, K = wq.shape
    assert N == N2
    dx = np.empty((M, K), dtype=np.float32)
    lib().oracle_linear_bwd_dx(_p(dy, _f32p), _p(wq, _i8p), float(s_w), _p(dx, _f32p), M, N, K)
    return dx


def linear_bwd_dw(dy, xq, s_x: float) -> np.ndarray:
    dy, xq = _f32(dy), _i8(xq)
    M, N = dy.shape
    M2, K = xq.shape
    assert M == M2
    dw = np.empty((N, K), dtype=np.float32)
    lib().oracle_linear_bwd_dw(_p(dy, _f32p), _p(xq, _i8p), float(s_x), _p(dw, _f32p), M, N, K)
    return dw


def linear_bwd_dx_at(dy, wq, s_w, idx_m, idx_k) -> np.ndarray:
    dy, wq = _f32(dy), _i8(wq)
    M, N = dy.shape
    K = wq.shape[1]
    im = np.ascontiguousarray(idx_m, dtype=np.int64)
    ik = np.ascontiguousarray(idx_k, dtype=np.int64)
    out = np.empty(im.size, dtype=np.float32)
    lib().oracle_linear_bwd_dx_at(_p(dy, _f32p), _p(wq, _i8p), float(s_w), M, N, K,
                                  _p(im, _i64p), _p(ik, _i64p), im.size, _p(out, _f32p))
    return out


def linear_bwd_dw_at(dy, xq, s_x, idx_n, idx_k) -> np.ndarray:
    dy, xq = _f32(dy), _i8(xq)
    M, N = dy.shape
    K = xq.shape[1]
    i_n = np.ascontiguousarray(idx_n, dtype=np.int64)
    ik = np.ascontiguousarray(idx_k, dtype=np.int64)
    out = np.empty(i_n.size, dtype=np.float32)
    lib().oracle_linear_bwd_dw_at(_p(dy, _f32p), _p(xq, _i8p), float(s_x), M, N, K,
                                  _p(i_n, _i64p), _p(ik, _i64p), i_n.size, _p(out, _f32p))
    return out


def grad_accum(acc, g) -> np.ndarray:
    """Returns acc (+) g as a new array (inputs untouched)."""
    out = _f32(acc).copy()
    g = _f32(g)
    assert out.size == g.size
    lib().oracle_grad_accum(_p(out, _f32p), _p(g, _f32p), out.size)
    return out


def running_sum(parts) -> np.ndarray:
    """Left fold of equal-length float32 arrays in the given order."""
    arrs = [_f32(p).ravel() for p in parts]
    S = len(arrs)
    n = arrs[0].size
    assert all(a.size == n for a in arrs)
    ptrs = (_f32p * S)(*[_p(a, _f32p) for a in arrs])
    out = np.empty(n, dtype=np.float32)
    lib().oracle_running_sum(ptrs, S, n, _p(out, _f32p))
    return out


def treefold_one(vals) -> np.float32:
    v = _f32(vals).ravel()
    return np.float32(lib().oracle_treefold_one(_p(v, _f32p), v.size))


def treefold_all_ranks(vals) -> np.ndarray:
    v = _f32(vals).ravel()
    out = np.empty(v.size, dtype=np.float32)
    lib().oracle_treefold_all_ranks(_p(v, _f32p), v.size, _p(out, _f32p))
    return out


def treefold(parts) -> np.ndarray:
    """parts: a sequence of R equal-length float32 arrays (any memory layout)."""
    arrs = [_f32(p).ravel() for p in parts]
    R = len(arrs)
    n = arrs[0].size
    assert all(a.size == n for a in arrs)
    ptrs = (_f32p * R)(*[_p(a, _f32p) for a in arrs])
    out = np.empty(n, dtype=np.float32)
    lib().oracle_treefold(ptrs, R, n, _p(out, _f32p))
    return out


def sumsq(g) -> np.float32:
    g = _f32(g).ravel()
    return np.float32(lib().oracle_sumsq(_p(g, _f32p), g.size))


def pow_t(b: float, t: int) -> np.float32:
    return np.float32(lib().oracle_pow_t(float(b), int(t)))


def clip_coef(s: float, max_norm: float) -> np.float32:
    return np.float32(lib().oracle_clip_coef(float(s), float(max_norm)))


def adamw_step(p, m, v, g, s: float, t: int, lr=4.5e-4, beta1=0.9, beta2=0.95, eps=1e-8,
               weight_decay=0.1, max_norm=1.0):
    """Returns new (p, m, v) as float32 arrays (inputs untouched)."""
    p, m, v = _f32(p).copy(), _f32(m).copy(), _f32(v).copy()
    g = _f32(g)
    hp = AdamWHparams(lr, beta1, beta2, eps, weight_decay, max_norm)
    lib().oracle_adamw_step(_p(p, _f32p), _p(m, _f32p), _p(v, _f32p), _p(g, _f32p), p.size,
                            float(s), ctypes.byref(hp), int(t))
    return p, m, v


def threads() -> int:
    return int(lib().oracle_threads())


def set_threads(n: int) -> None:
    """Threads of the parallel loops over output elements (bits unchanged)."""
    lib().oracle_set_threads(int(n))


# ---------------------------------------------------------------- attention

def exp(x: float) -> np.float32:
    """The softmax's e^x (Cody-Waite reduction + degree-7 Taylor, binary32)."""
    return np.float32(lib().oracle_exp(float(x)))


def attn_quant_p(p: float) -> int:
    return int(lib().oracle_attn_quant_p(float(p)))


def attn_fx(x: float) -> int:
    return int(lib().oracle_attn_fx(float(x)))


def attn_fix2f(a: int) -> np.float32:
    return np.float32(lib().oracle_attn_fix2f(int(a)))


def _attn_shapes(q, k):
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, T, Hkv, D) and Hq % Hkv == 0
    return B, T, Hq, Hkv, D


def attn_fwd(q, k, vq, s_v: float, W: int):
    """q [B,T,Hq,D], k and vq [B,T,Hkv,D] -> (o [B,T,Hq,D], m [B,T,Hq], l [B,T,Hq])."""
    q, k, vq = _f32(q), _f32(k), _i8(vq)
    B, T, Hq, Hkv, D = _attn_shapes(q, k)
    o = np.empty((B, T, Hq, D), np.float32)
    m = np.empty((B, T, Hq), np.float32)
    l = np.empty((B, T, Hq), np.float32)
    lib().oracle_attn_fwd(_p(q, _f32p), _p(k, _f32p), _p(vq, _i8p), float(s_v), _p(o, _f32p),
                          _p(m, _f32p), _p(l, _f32p), B, T, Hq, Hkv, D, int(W))
    return o, m, l


def attn_fwd_rows(q, k, vq, s_v: float, W: int, rows):
    """Rows given as flat (b, i, h) indices -> (o [n,D], m [n], l [n])."""
    q, k, vq = _f32(q), _f32(k), _i8(vq)
    B, T, Hq, Hkv, D = _attn_shapes(q, k)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    o = np.empty((n, D), np.float32)
    m = np.empty(n, np.float32)
    l = np.empty(n, np.float32)
    lib().oracle_attn_fwd_rows(_p(q, _f32p), _p(k, _f32p), _p(vq, _i8p), float(s_v),
                               _p(rows, _i64p), n, _p(o, _f32p), _p(m, _f32p), _p(l, _f32p),
                               B, T, Hq, Hkv, D, int(W))
    return o, m, l


def attn_bwd(q, k, vq, s_v: float, o, dout, m, l, W: int):
    """-> (dq [B,T,Hq,D], dk [B,T,Hkv,D], dv [B,T,Hkv,D])."""
    q, k, vq, o, dout, m, l = _f32(q), _f32(k), _i8(vq), _f32(o), _f32(dout), _f32(m), _f32(l)
    B, T, Hq, Hkv, D = _attn_shapes(q, k)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(k)
    lib().oracle_attn_bwd(_p(q, _f32p), _p(k, _f32p), _p(vq, _i8p), float(s_v), _p(o, _f32p),
                          _p(dout, _f32p), _p(m, _f32p), _p(l, _f32p), _p(dq, _f32p),
                          _p(dk, _f32p), _p(dv, _f32p), B, T, Hq, Hkv, D, int(W))
    return dq, dk, dv


def attn_bwd_rows(q, k, vq, s_v: float, o, dout, m, l, W: int, qrows, krows):
    """dq for flat (b, i, h) rows qrows, dk and dv for flat (b, j, g) rows krows."""
    q, k, vq, o, dout, m, l = _f32(q), _f32(k), _i8(vq), _f32(o), _f32(dout), _f32(m), _f32(l)
    B, T, Hq, Hkv, D = _attn_shapes(q, k)
    qrows = np.ascontiguousarray(qrows, dtype=np.int64)
    krows = np.ascontiguousarray(krows, dtype=np.int64)
    dq = np.empty((qrows.size, D), np.float32)
    dk = np.empty((krows.size, D), np.float32)
    dv = np.empty((krows.size, D), np.float32)
    lib().oracle_attn_bwd_rows(_p(q, _f32p), _p(k, _f32p), _p(vq, _i8p), float(s_v),
                               _p(o, _f32p), _p(dout, _f32p), _p(m, _f32p), _p(l, _f32p),
                               _p(qrows, _i64p), qrows.size, _p(dq, _f32p), _p(krows, _i64p),
                               krows.size, _p(dk, _f32p), _p(dv, _f32p), B, T, Hq, Hkv, D,
                               int(W))
    return dq, dk, dv


from .merkle import LEAF_BYTES as HASH_LEAF_BYTES, state_hash, mth, audit_path  # noqa: E402,F401
