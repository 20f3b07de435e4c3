"""Thin Python binding of librepro.so (include/repro.h): argument marshalling
only.  Every step of the path runs in the library's CUDA kernels; torch is used
for device memory and streams.  There is no fallback: if the library is not
built, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librepro.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "repro.h")

REPRO_OK = 0
STATUS_NAMES = {
    0: "REPRO_OK", -1: "REPRO_ERR_ARG", -2: "REPRO_ERR_SHAPE", -3: "REPRO_ERR_ALIGN",
    -4: "REPRO_ERR_ARCH", -5: "REPRO_ERR_LAUNCH", -6: "REPRO_ERR_TIMEOUT",
    -7: "REPRO_ERR_WORKSPACE", -8: "REPRO_ERR_ALIAS", -9: "REPRO_ERR_SELFTEST",
    -10: "REPRO_ERR_NONFINITE",
}
REPRO_ERR_TIMEOUT = -6
REPRO_ERR_NONFINITE = -10
REPRO_DEBUG_CHECK_FINITE = 1
REPRO_SCALE_WEIGHT_MEANABS = 0
REPRO_SCALE_ACT_AMAX = 1
REPRO_BWD_DW_ACCUMULATE = 1
REPRO_QMAX = 127
REPRO_MAX_REPLICAS = 64


class ReproError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)} "
                         f"({lib().repro_status_str(status).decode()})")


class AdamWHparams(ctypes.Structure):
    _fields_ = [(k, ctypes.c_float) for k in
                ("lr", "beta1", "beta2", "eps", "weight_decay", "max_norm")]


class LaunchCfg(ctypes.Structure):
    _fields_ = [("bwd_segment_log2", ctypes.c_int), ("reduce_block_log2", ctypes.c_int),
                ("fwd_path", ctypes.c_int), ("elementwise_blocks", ctypes.c_int),
                ("bwd_kernel", ctypes.c_int), ("fwd_selftest", ctypes.c_int)]


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_sz = ctypes.c_size_t

_SIGNATURES = {
    "repro_wscale": (_int, [_vp, _i64, _int, _int, _vp, _vp, _sz, _vp]),
    "repro_wscale_ws_bytes": (_sz, [_i64]),
    "repro_wscale_noalloc": (_int, [_vp, _i64, _int, _int, _vp, _vp]),
    "repro_quant_i8": (_int, [_vp, _i64, _vp, _int, _vp, _vp]),
    "repro_wscale_multi": (_int, [ctypes.POINTER(_vp), ctypes.POINTER(_i64), _int, _int, _int,
                                  _vp, _vp, _sz, _vp]),
    "repro_wscale_multi_ws_bytes": (_sz, [ctypes.POINTER(_i64), _int]),
    "repro_quant_i8_multi": (_int, [ctypes.POINTER(_vp), ctypes.POINTER(_i64), _int, _vp, _int,
                                    ctypes.POINTER(_vp), _vp]),
    "repro_linear_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _vp]),
    "repro_linear_fwd_ws_bytes": (_sz, [_i64, _i64, _i64]),
    "repro_linear_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int,
                                _vp, _sz, _vp]),
    "repro_linear_bwd_ws_bytes": (_sz, [_i64, _i64, _i64]),
    "repro_grad_accum": (_int, [_vp, _vp, _i64, _vp]),
    "repro_treefold": (_int, [ctypes.POINTER(_vp), _int, _i64, _vp, _vp]),
    "repro_running_sum": (_int, [ctypes.POINTER(_vp), _int, _i64, _vp, _vp]),
    "repro_sumsq": (_int, [_vp, _i64, _vp, _vp, _sz, _vp]),
    "repro_sumsq_ws_bytes": (_sz, [_i64]),
    "repro_adamw_step": (_int, [_vp, _vp, _vp, _vp, _i64, _vp, ctypes.POINTER(AdamWHparams),
                                _i64, _vp]),
    "repro_state_hash": (_int, [ctypes.POINTER(_vp), ctypes.POINTER(_i64), _int, _vp, _vp, _sz,
                                _vp]),
    "repro_state_hash_ws_bytes": (_sz, [ctypes.POINTER(_i64), _int]),
    "repro_attn_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                              _i64, _vp, _sz, _vp]),
    "repro_attn_fwd_ws_bytes": (_sz, [_i64, _i64, _i64, _i64]),
    "repro_attn_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                              _i64, _i64, _i64, _i64, _vp, _sz, _vp, _sz, _vp]),
    "repro_attn_bwd_ws_bytes": (_sz, [_i64, _i64, _i64, _i64]),
    "repro_selftest": (_int, [_vp, _sz, _vp]),
    "repro_selftest_ws_bytes": (_sz, []),
    "repro_status_str": (ctypes.c_char_p, [_int]),
    "repro_version": (_int, []),
    "repro_device_check": (_int, [_vp]),
    "repro_wait_probe": (_int, [_int, _vp]),
    "repro_launch_count": (ctypes.c_uint64, []),
    "repro_set_launch_cfg": (_int, [ctypes.POINTER(LaunchCfg)]),
    "repro_set_debug": (_int, [_int]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "bitwise_reproducible_int8_gb300.build_lib.build() (there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def declared_functions() -> list:
    """Names of the functions declared in include/repro.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int|size_t|uint64_t)\s+(repro_\w+)\s*\(",
                                 text, flags=re.M)))


# ------------------------------------------------------------------ marshalling

def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _check(fn: str, status: int) -> None:
    if status != REPRO_OK:
        raise ReproError(fn, status)


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ the calls

def repro_wscale_ws_bytes(n: int) -> int:
    return int(lib().repro_wscale_ws_bytes(int(n)))


def repro_wscale(x: torch.Tensor, mode: int, scale_out: torch.Tensor, ws=None,
                 qmax: int = REPRO_QMAX, stream=None) -> None:
    """scale_out[0] <- weight (mode 0) or activation (mode 1) scale of x."""
    n = x.numel()
    if ws is None:
        ws = _workspace(repro_wscale_ws_bytes(n), x.device)
    _check("repro_wscale", lib().repro_wscale(
        _ptr(x, torch.float32, "x"), n, int(mode), int(qmax),
        _ptr(scale_out, torch.float32, "scale_out"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 1 << 62,
        _stream(stream)))


def repro_wscale_noalloc(x: torch.Tensor, mode: int, scale_out: torch.Tensor,
                         qmax: int = REPRO_QMAX, stream=None) -> None:
    """repro_wscale without a workspace, for callers that cannot allocate
    device memory; scratch comes from a fixed array inside the library."""
    _check("repro_wscale_noalloc", lib().repro_wscale_noalloc(
        _ptr(x, torch.float32, "x"), x.numel(), int(mode), int(qmax),
        _ptr(scale_out, torch.float32, "scale_out"), _stream(stream)))


def repro_quant_i8(x: torch.Tensor, scale: torch.Tensor, q_out: torch.Tensor,
                   qmax: int = REPRO_QMAX, stream=None) -> None:
    if q_out.numel() != x.numel():
        raise ValueError("q_out must have as many elements as x")
    _check("repro_quant_i8", lib().repro_quant_i8(
        _ptr(x, torch.float32, "x"), x.numel(), _ptr(scale, torch.float32, "scale"), int(qmax),
        _ptr(q_out, torch.int8, "q_out"), _stream(stream)))


def _tables(tensors, dtype, name):
    n = len(tensors)
    ptrs = (_vp * max(n, 1))(*[_ptr(t, dtype, name) for t in tensors])
    sizes = (_i64 * max(n, 1))(*[int(t.numel()) for t in tensors])
    return ptrs, sizes


def repro_wscale_multi_ws_bytes(sizes) -> int:
    arr = (_i64 * max(len(sizes), 1))(*[int(v) for v in sizes])
    return int(lib().repro_wscale_multi_ws_bytes(arr, len(sizes)))


def repro_wscale_multi(xs, mode: int, scales_out: torch.Tensor, ws=None,
                       qmax: int = REPRO_QMAX, stream=None) -> None:
    """scales_out[t] <- the scale of xs[t] (mode 0 weight, 1 activation) for
    every t, in one pass; the bits of repro_wscale on each tensor."""
    ptrs, sizes = _tables(xs, torch.float32, "x")
    if scales_out.numel() < len(xs):
        raise ValueError("scales_out needs one float per tensor")
    if ws is None:
        ws = _workspace(repro_wscale_multi_ws_bytes([x.numel() for x in xs]), xs[0].device)
    _check("repro_wscale_multi", lib().repro_wscale_multi(
        ptrs, sizes, len(xs), int(mode), int(qmax), _ptr(scales_out, torch.float32, "scales_out"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def repro_quant_i8_multi(xs, scales: torch.Tensor, q_outs, qmax: int = REPRO_QMAX,
                         stream=None) -> None:
    """q_outs[t] <- int8 codes of xs[t] with scales[t], every t in one launch."""
    if len(q_outs) != len(xs) or any(q.numel() != x.numel() for q, x in zip(q_outs, xs)):
        raise ValueError("one q_out of x's size per tensor")
    ptrs, sizes = _tables(xs, torch.float32, "x")
    qptrs, _ = _tables(q_outs, torch.int8, "q_out")
    _check("repro_quant_i8_multi", lib().repro_quant_i8_multi(
        ptrs, sizes, len(xs), _ptr(scales, torch.float32, "scales"), int(qmax), qptrs,
        _stream(stream)))


def repro_linear_fwd_ws_bytes(M: int, N: int, K: int) -> int:
    return int(lib().repro_linear_fwd_ws_bytes(int(M), int(N), int(K)))


def repro_linear_fwd(xq: torch.Tensor, wq: torch.Tensor, s_x: torch.Tensor, s_w: torch.Tensor,
                     y: torch.Tensor, ws=None, stream=None) -> None:
    M, K = xq.shape
    N, K2 = wq.shape
    if K != K2 or tuple(y.shape) != (M, N):
        raise ValueError("shape mismatch: xq [M,K], wq [N,K], y [M,N]")
    if ws is None:
        need = repro_linear_fwd_ws_bytes(M, N, K)
        ws = _workspace(need, y.device) if need > 0 else None
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check("repro_linear_fwd", lib().repro_linear_fwd(
        _ptr(xq, torch.int8, "xq"), _ptr(wq, torch.int8, "wq"), _ptr(s_x, torch.float32, "s_x"),
        _ptr(s_w, torch.float32, "s_w"), _ptr(y, torch.float32, "y"), M, N, K,
        _ptr(ws, None, "ws"), ws_bytes, _stream(stream)))


def repro_linear_bwd_ws_bytes(M: int, N: int, K: int) -> int:
    return int(lib().repro_linear_bwd_ws_bytes(int(M), int(N), int(K)))


def repro_linear_bwd(dy: torch.Tensor, xq, wq, s_x, s_w, dx=None, dw=None,
                     accumulate: bool = False, ws=None, stream=None) -> None:
    M, N = dy.shape
    K = (xq if xq is not None else wq).shape[1]
    if dx is not None and tuple(dx.shape) != (M, K):
        raise ValueError("dx must be [M,K]")
    if dw is not None and tuple(dw.shape) != (N, K):
        raise ValueError("dw must be [N,K]")
    if ws is None:
        need = repro_linear_bwd_ws_bytes(M, N, K)
        ws = _workspace(need, dy.device) if need > 0 else None
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check("repro_linear_bwd", lib().repro_linear_bwd(
        _ptr(dy, torch.float32, "dy"), _ptr(xq, torch.int8, "xq"), _ptr(wq, torch.int8, "wq"),
        _ptr(s_x, torch.float32, "s_x"), _ptr(s_w, torch.float32, "s_w"),
        _ptr(dx, torch.float32, "dx"), _ptr(dw, torch.float32, "dw"), M, N, K,
        REPRO_BWD_DW_ACCUMULATE if accumulate else 0, _ptr(ws, None, "ws"), ws_bytes,
        _stream(stream)))


def repro_grad_accum(acc: torch.Tensor, g: torch.Tensor, stream=None) -> None:
    if acc.numel() != g.numel():
        raise ValueError("acc and g must have the same number of elements")
    _check("repro_grad_accum", lib().repro_grad_accum(
        _ptr(acc, torch.float32, "acc"), _ptr(g, torch.float32, "g"), acc.numel(),
        _stream(stream)))


def repro_running_sum(parts, out: torch.Tensor, stream=None) -> None:
    """out <- left fold of the partials in the given (mesh) order."""
    S = len(parts)
    n = out.numel()
    if any(p.numel() != n for p in parts):
        raise ValueError("every partial must have out.numel() elements")
    arr = (_vp * max(S, 1))(*[_ptr(p, torch.float32, "part") for p in parts])
    _check("repro_running_sum", lib().repro_running_sum(arr, S, n, _ptr(out, torch.float32, "out"),
                                                        _stream(stream)))


def repro_treefold(parts, out: torch.Tensor, stream=None) -> None:
    R = len(parts)
    n = out.numel()
    if any(p.numel() != n for p in parts):
        raise ValueError("every partial must have out.numel() elements")
    arr = (_vp * max(R, 1))(*[_ptr(p, torch.float32, "part") for p in parts])
    _check("repro_treefold", lib().repro_treefold(arr, R, n, _ptr(out, torch.float32, "out"),
                                                  _stream(stream)))


def repro_attn_fwd_ws_bytes(B: int, T: int, Hq: int, W: int = 0) -> int:
    return int(lib().repro_attn_fwd_ws_bytes(int(B), int(T), int(Hq), int(W)))


def repro_attn_fwd(q: torch.Tensor, k: torch.Tensor, vq: torch.Tensor, s_v: torch.Tensor,
                   o: torch.Tensor, m: torch.Tensor, l: torch.Tensor, W: int = 0, ws=None,
                   stream=None) -> None:
    """q, o [B,T,Hq,128] fp32; k [B,T,Hkv,128] fp32; vq [B,T,Hkv,128] int8;
    s_v [1]; m, l [B,T,Hq] outputs.  W: sliding window (0: full causal).
    ws: optional logit cache of repro_attn_fwd_ws_bytes bytes (None: the
    second pass recomputes the logits; same bits)."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check("repro_attn_fwd", lib().repro_attn_fwd(
        _ptr(q, torch.float32, "q"), _ptr(k, torch.float32, "k"), _ptr(vq, torch.int8, "vq"),
        _ptr(s_v, torch.float32, "s_v"), _ptr(o, torch.float32, "o"),
        _ptr(m, torch.float32, "m"), _ptr(l, torch.float32, "l"), B, T, Hq, Hkv, D, int(W),
        _ptr(ws, None, "ws"), ws_bytes, _stream(stream)))


def repro_attn_bwd_ws_bytes(B: int, T: int, Hq: int, W: int = 0) -> int:
    """Workspace of repro_attn_bwd for window W; W = -1: a call without the
    forward's cache."""
    return int(lib().repro_attn_bwd_ws_bytes(int(B), int(T), int(Hq), int(W)))


def repro_attn_bwd(q, k, vq, s_v, o, dout, m, l, dq, dk, dv, W: int = 0, ws=None,
                   fwd_ws=None, stream=None) -> None:
    """dq [B,T,Hq,128], dk and dv [B,T,Hkv,128] from the forward's inputs,
    output o, row statistics m, l and the upstream gradient dout.  fwd_ws:
    optionally the logit cache repro_attn_fwd filled for these inputs."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if ws is None:
        ws = _workspace(repro_attn_bwd_ws_bytes(B, T, Hq, int(W) if fwd_ws is not None else -1),
                        q.device)
    f32 = torch.float32
    _check("repro_attn_bwd", lib().repro_attn_bwd(
        _ptr(q, f32, "q"), _ptr(k, f32, "k"), _ptr(vq, torch.int8, "vq"), _ptr(s_v, f32, "s_v"),
        _ptr(o, f32, "o"), _ptr(dout, f32, "dout"), _ptr(m, f32, "m"), _ptr(l, f32, "l"),
        _ptr(dq, f32, "dq"), _ptr(dk, f32, "dk"), _ptr(dv, f32, "dv"), B, T, Hq, Hkv, D, int(W),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(fwd_ws, None, "fwd_ws"),
        fwd_ws.numel() * fwd_ws.element_size() if fwd_ws is not None else 0, _stream(stream)))


def repro_selftest(device=None, stream=None) -> int:
    """Runs the tensor-core forward's exactness self-test; returns the status
    (REPRO_OK when every output matches the exact CUDA-core path)."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    ws = _workspace(int(lib().repro_selftest_ws_bytes()), dev)
    return int(lib().repro_selftest(_ptr(ws, None, "ws"), ws.numel(), _stream(stream)))


REPRO_HASH_LEAF_BYTES = 4096


def _hash_tables(buffers):
    nb = len(buffers)
    ptrs = (_vp * max(nb, 1))(*[_ptr(b, None, "buffer") if b.numel() else None for b in buffers])
    sizes = (_i64 * max(nb, 1))(*[b.numel() * b.element_size() for b in buffers])
    return ptrs, sizes, nb


def repro_state_hash_ws_bytes(buffers) -> int:
    """Workspace for hashing these tensors (their bytes, in order)."""
    _, sizes, nb = _hash_tables(buffers)
    return int(lib().repro_state_hash_ws_bytes(sizes, nb))


def repro_state_hash(buffers, digest: torch.Tensor, ws=None, stream=None) -> None:
    """digest (32 uint8, device) <- Merkle Tree Hash of the tensors' bytes."""
    for b in buffers:
        if not b.is_contiguous():
            raise ValueError("state buffers must be contiguous")
    ptrs, sizes, nb = _hash_tables(buffers)
    if digest.numel() != 32 or digest.dtype != torch.uint8:
        raise ValueError("digest must be 32 uint8")
    if ws is None:
        ws = _workspace(int(lib().repro_state_hash_ws_bytes(sizes, nb)), digest.device)
    _check("repro_state_hash", lib().repro_state_hash(
        ptrs, sizes, nb, _ptr(digest, torch.uint8, "digest"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)))


def repro_sumsq_ws_bytes(n: int) -> int:
    return int(lib().repro_sumsq_ws_bytes(int(n)))


def repro_sumsq(g: torch.Tensor, out: torch.Tensor, ws=None, stream=None) -> None:
    """out[0] <- canonical sum of g_i (x) g_i."""
    n = g.numel()
    if ws is None:
        ws = _workspace(repro_sumsq_ws_bytes(n), g.device)
    _check("repro_sumsq", lib().repro_sumsq(
        _ptr(g, torch.float32, "g"), n, _ptr(out, torch.float32, "out"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)))


def repro_adamw_step(p: torch.Tensor, m: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                     sumsq: torch.Tensor, t: int, lr: float = 4.5e-4, beta1: float = 0.9,
                     beta2: float = 0.95, eps: float = 1e-8, weight_decay: float = 0.1,
                     max_norm: float = 1.0, stream=None) -> None:
    """Clip to the global norm sqrt(sumsq) and apply AdamW step t in place."""
    n = p.numel()
    if not (m.numel() == v.numel() == g.numel() == n):
        raise ValueError("p, m, v and g must have the same number of elements")
    hp = AdamWHparams(lr, beta1, beta2, eps, weight_decay, max_norm)
    _check("repro_adamw_step", lib().repro_adamw_step(
        _ptr(p, torch.float32, "p"), _ptr(m, torch.float32, "m"), _ptr(v, torch.float32, "v"),
        _ptr(g, torch.float32, "g"), n, _ptr(sumsq, torch.float32, "sumsq"), ctypes.byref(hp),
        int(t), _stream(stream)))


def repro_status_str(status: int) -> str:
    return lib().repro_status_str(int(status)).decode()


def repro_version() -> int:
    return int(lib().repro_version())


def repro_launch_count() -> int:
    return int(lib().repro_launch_count())


def repro_device_check(stream=None) -> int:
    return int(lib().repro_device_check(_stream(stream)))


def repro_wait_probe(arrive: int, stream=None) -> int:
    """Enqueue the bounded-wait probe; arrive=0 makes the wait run out."""
    return int(lib().repro_wait_probe(int(arrive), _stream(stream)))


def repro_set_debug(flags: int) -> None:
    """Debug checks (REPRO_DEBUG_CHECK_FINITE: scan every float input; a NaN or
    an infinity makes the next repro_device_check return REPRO_ERR_NONFINITE)."""
    _check("repro_set_debug", lib().repro_set_debug(int(flags)))


def repro_set_launch_cfg(bwd_segment_log2: int = -1, reduce_block_log2: int = -1,
                         fwd_path: int = -1, elementwise_blocks: int = -1, bwd_kernel: int = -1,
                         fwd_selftest: int = -1, reset: bool = False):
    if reset:
        _check("repro_set_launch_cfg", lib().repro_set_launch_cfg(None))
        return
    cfg = LaunchCfg(bwd_segment_log2, reduce_block_log2, fwd_path, elementwise_blocks, bwd_kernel,
                    fwd_selftest)
    _check("repro_set_launch_cfg", lib().repro_set_launch_cfg(ctypes.byref(cfg)))
