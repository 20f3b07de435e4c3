"""Host-side tests of the C ABI (no GPU needed): the library loads and exports
every function include/repro.h declares; invalid arguments are rejected with
the documented status codes before anything is launched; workspace sizes and
the launch-configuration hook behave as documented."""
import ctypes

import pytest

from bitwise_reproducible_int8_gb300 import build_lib, repro


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return repro.lib()


A = 0x10000  # a fake, 16-byte aligned device address (never dereferenced)


def test_exports_every_declared_symbol(L):
    names = repro.declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    for n in ["repro_wscale", "repro_quant_i8", "repro_linear_fwd", "repro_linear_bwd",
              "repro_grad_accum", "repro_treefold"]:
        assert n in names


def test_status_strings_and_version(L):
    assert repro.repro_version() == 1
    for code in range(-10, 1):
        assert repro.repro_status_str(code) != "unknown status"
    assert repro.repro_status_str(-99) == "unknown status"


def test_debug_flags(L):
    assert L.repro_set_debug(2) == -1 and L.repro_set_debug(-1) == -1   # unknown flags
    assert L.repro_set_debug(repro.REPRO_DEBUG_CHECK_FINITE) == 0
    # invalid arguments are still rejected before anything (a scan included) is enqueued
    assert L.repro_wscale(None, 10, 0, 127, A, A * 4, 1 << 20, None) == -1
    assert L.repro_set_debug(0) == 0
    assert repro.STATUS_NAMES[-10] == "REPRO_ERR_NONFINITE"


def test_wscale_argument_checks(L):
    f = L.repro_wscale
    ws = A * 4
    assert f(None, 10, 0, 127, A, ws, 1 << 20, None) == -1           # null x
    assert f(A, 10, 2, 127, A + 64, ws, 1 << 20, None) == -1         # bad mode
    assert f(A, 10, 0, 100, A + 64, ws, 1 << 20, None) == -1         # q_max
    assert f(A, 0, 0, 127, A + 64, ws, 1 << 20, None) == -2          # empty
    assert f(A + 4, 10, 0, 127, A + 64, ws, 1 << 20, None) == -3     # misaligned x
    assert f(A, 10, 0, 127, A + 64, None, 0, None) == -7             # no workspace
    assert f(A, 1 << 20, 0, 127, A + 64, ws, 16, None) == -7         # small workspace
    assert f(A, 100, 0, 127, A + 64, A, 1 << 20, None) == -8         # ws overlaps x


def test_wscale_ws_bytes_covers_all_blocks(L):
    for n in [1, 64, 65, 10 ** 6, 23068672]:
        C = (n + 63) // 64
        assert repro.repro_wscale_ws_bytes(n) >= 4 * (C + (C + 1) // 2)
    assert repro.repro_wscale_ws_bytes(0) == 0


def test_multi_tensor_argument_checks(L):
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    B = 1 << 32
    xs = (P * 3)(B, B * 2, B * 3)
    ns = (I64 * 3)(100, 64, 4097)
    need = repro.repro_wscale_multi_ws_bytes([100, 64, 4097])
    assert need >= 4 * (2 + 1 + 65)
    assert repro.repro_wscale_multi_ws_bytes([100, 0]) == 0
    assert repro.repro_wscale_multi_ws_bytes([]) == 0
    f = L.repro_wscale_multi
    ws = B * 8
    assert f(xs, ns, 0, 0, 127, B * 4, ws, need, None) == -1            # no tensors
    assert f(xs, ns, 65, 0, 127, B * 4, ws, need, None) == -1           # too many
    assert f(xs, ns, 3, 2, 127, B * 4, ws, need, None) == -1            # mode
    assert f(xs, ns, 3, 0, 126, B * 4, ws, need, None) == -1            # q_max
    assert f(xs, (I64 * 3)(100, 0, 5), 3, 0, 127, B * 4, ws, need, None) == -2
    assert f((P * 3)(B, B * 2 + 4, B * 3), ns, 3, 0, 127, B * 4, ws, need, None) == -3
    assert f(xs, ns, 3, 0, 127, B * 4, ws, need - 4, None) == -7        # small workspace
    assert f(xs, ns, 3, 0, 127, B * 2 + 8, ws, need, None) == -8        # scales inside x[1]
    assert f(xs, ns, 3, 0, 127, B * 4, B * 3, need, None) == -8         # ws overlaps x[2]
    assert f(xs, ns, 3, 0, 127, B * 4, ws, need, None) not in (-1, -2, -3, -7, -8)
    g = L.repro_quant_i8_multi
    qs = (P * 3)(B * 5, B * 6, B * 7)
    assert g(xs, ns, 3, B * 4, 126, qs, None) == -1
    assert g(xs, (I64 * 3)(1, -1, 1), 3, B * 4, 127, qs, None) == -2
    assert g(xs, ns, 3, B * 4, 127, (P * 3)(B * 5, B * 6 + 8, B * 7), None) == -3
    assert g(xs, ns, 3, B * 4, 127, (P * 3)(B * 5, B * 5 + 64, B * 7), None) == -8   # q0, q1 overlap
    assert g(xs, ns, 3, B * 4, 127, (P * 3)(B * 5, B * 2, B * 7), None) == -8        # q1 over x1
    assert g(xs, (I64 * 3)(0, 0, 0), 3, B * 4, 127, qs, None) == 0       # nothing to do
    assert g(xs, ns, 3, B * 4, 127, qs, None) not in (-1, -2, -3, -8)


def test_quant_argument_checks(L):
    f = L.repro_quant_i8
    assert f(A, 10, A + 4096, 126, A * 2, None) == -1
    assert f(A, -1, A + 4096, 127, A * 2, None) == -2
    assert f(None, 0, None, 127, None, None) == 0                     # empty is a no-op
    assert f(None, 10, A + 4096, 127, A * 2, None) == -1
    assert f(A, 10, A + 4096, 127, A * 2 + 8, None) == -3             # misaligned q
    assert f(A, 10, A + 4096, 127, A + 8, None) == -3
    assert f(A, 100, A + 4096, 127, A + 16, None) == -8               # q inside x


def test_linear_fwd_argument_checks(L):
    def f(*a):
        return L.repro_linear_fwd(*a[:8], None, 0, None)
    assert f(A, A * 2, A * 3, A * 3 + 4, A * 4, 8, 8, 133145) == -2   # K too large
    assert f(A, A * 2, A * 3, A * 3 + 4, A * 4, -1, 8, 8) == -2
    assert f(None, None, None, None, None, 0, 8, 8) == 0              # M == 0
    assert f(A, A * 2, None, A * 3, A * 4, 8, 8, 8) == -1             # null scale
    assert f(A + 1, A * 2, A * 3, A * 3 + 4, A * 4, 8, 8, 8) == -3
    assert f(A, A * 2, A * 3, A * 3 + 4, A, 8, 8, 8) == -8            # y overlaps xq


def test_linear_fwd_workspace(L):
    try:
        repro.repro_set_launch_cfg(fwd_path=0)
        assert repro.repro_linear_fwd_ws_bytes(16384, 2048, 2048) == 0
        repro.repro_set_launch_cfg(fwd_path=1)
        need = repro.repro_linear_fwd_ws_bytes(16384, 2048, 2048)
        assert need >= 2 * (16384 + 2048) * 2048
        # small tensor-core shapes still leave room for the once-per-device
        # exactness check the first call runs in the workspace
        assert repro.repro_linear_fwd_ws_bytes(8, 8, 8) == L.repro_selftest_ws_bytes()
        assert repro.repro_linear_fwd_ws_bytes(16, 16, 12) == 0     # K % 8 != 0: CUDA cores
        B = 1 << 32
        assert L.repro_linear_fwd(B, B * 2, B * 3, B * 3 + 4, B * 4, 16384, 2048, 2048,
                                  None, 0, None) == -7
        assert L.repro_linear_fwd(B, B * 2, B * 3, B * 3 + 4, B * 4, 16384, 2048, 2048,
                                  B * 8, need - 1, None) == -7
        assert L.repro_linear_fwd(B, B * 2, B * 3, B * 3 + 4, B * 4, 16384, 2048, 2048,
                                  B, need, None) == -8              # ws overlaps xq
    finally:
        repro.repro_set_launch_cfg(reset=True)


def test_linear_bwd_argument_checks(L):
    f = L.repro_linear_bwd
    M = N = K = 8
    args = lambda **k: [k.get("dy", A), k.get("xq", A * 2), k.get("wq", A * 3),  # noqa: E731
                        k.get("sx", A * 4), k.get("sw", A * 4 + 4), k.get("dx", A * 5),
                        k.get("dw", A * 6), M, N, K, k.get("flags", 0), None, 0, None]
    assert f(*args(flags=2)) == -1
    assert f(*args(dx=None, dw=None)) == -1
    assert f(*args(wq=None)) == -1                       # dx wanted, wq missing
    assert f(*args(xq=None)) == -1                       # dw wanted, xq missing
    assert f(*args(dy=A + 8)) == -3
    assert f(*args(dx=A)) == -8                          # dx overlaps dy
    assert f(*args(dw=A * 5)) == -8                      # dx and dw overlap


def test_bwd_workspace_follows_segments(L):
    try:
        repro.repro_set_launch_cfg(bwd_segment_log2=8, bwd_kernel=1)
        assert repro.repro_linear_bwd_ws_bytes(16384, 2048, 2048) == 0
        repro.repro_set_launch_cfg(bwd_segment_log2=4, bwd_kernel=1)
        # dW: 256 chunks / 16 = 16 segments of N x K partials
        assert repro.repro_linear_bwd_ws_bytes(16384, 2048, 2048) == 16 * 2048 * 2048 * 4
        f = L.repro_linear_bwd
        B = 1 << 32   # widely spaced fake addresses: nothing overlaps
        assert f(B, B * 2, B * 3, B * 4, B * 4 + 4, B * 5, B * 6, 16384, 8, 8, 0, None, 0,
                 None) == -7
        # the tensor-copy kernel adds its prepared operands after the partials:
        # max(dY^T + W^, dY + X^) = 2 * 16384 * 2048 floats here
        opnd = 2 * 16384 * 2048 * 4
        repro.repro_set_launch_cfg(bwd_segment_log2=8, bwd_kernel=8)
        assert repro.repro_linear_bwd_ws_bytes(16384, 2048, 2048) == opnd
        repro.repro_set_launch_cfg(bwd_segment_log2=4, bwd_kernel=8)
        assert repro.repro_linear_bwd_ws_bytes(16384, 2048, 2048) == 16 * 2048 * 2048 * 4 + opnd
        # the workspace may overlap no operand: the backward writes prepared
        # operands there before it reads xq / wq / the scales
        need = repro.repro_linear_bwd_ws_bytes(16384, 2048, 2048)
        args = [B, B * 2, B * 3, B * 4, B * 4 + 4, B * 5, B * 6, 16384, 2048, 2048, 0]
        assert f(*args, B * 8, need, None) != -8   # (no GPU here: arch or launch status)
        assert f(*args, B * 2, need, None) == -8   # ws overlaps xq
        assert f(*args, B * 3, need, None) == -8   # ws overlaps wq
        assert f(*args, B * 4 - 16, need, None) == -8   # ws overlaps s_x and s_w
        # rows that are not 16-byte aligned take the register-prefetch kernel: no operand region
        repro.repro_set_launch_cfg(bwd_segment_log2=8, bwd_kernel=8)
        assert repro.repro_linear_bwd_ws_bytes(64, 30, 20) == 0
    finally:
        repro.repro_set_launch_cfg(reset=True)


def test_grad_accum_and_treefold_checks(L):
    assert L.repro_grad_accum(A, A, 10, None) == -8
    assert L.repro_grad_accum(A, A + 16, 10, None) == -8
    assert L.repro_grad_accum(A + 4, A * 2, 10, None) == -3
    assert L.repro_grad_accum(None, None, 0, None) == 0
    P = ctypes.c_void_p
    parts = (P * 3)(A, A * 2, A * 3)
    assert L.repro_treefold(parts, 0, 10, A * 4, None) == -1
    assert L.repro_treefold(parts, 65, 10, A * 4, None) == -1
    assert L.repro_treefold(None, 3, 10, A * 4, None) == -1
    assert L.repro_treefold(parts, 3, 10, A * 2, None) == -8          # out overlaps parts[1]
    bad = (P * 3)(A, A * 2 + 4, A * 3)
    assert L.repro_treefold(bad, 3, 10, A * 4, None) == -3
    null = (P * 3)(A, None, A * 3)
    assert L.repro_treefold(null, 3, 10, A * 4, None) == -1


def test_launch_cfg_validation(L):
    try:
        with pytest.raises(repro.ReproError):
            repro.repro_set_launch_cfg(bwd_segment_log2=9)
        with pytest.raises(repro.ReproError):
            repro.repro_set_launch_cfg(reduce_block_log2=11)
        with pytest.raises(repro.ReproError):
            repro.repro_set_launch_cfg(fwd_path=3)
        for k in (0, 2, 7, 9):   # only the two shipped kernels, 1 and 8
            with pytest.raises(repro.ReproError):
                repro.repro_set_launch_cfg(bwd_kernel=k)
        repro.repro_set_launch_cfg(bwd_kernel=1)
        repro.repro_set_launch_cfg(bwd_kernel=8)
        for v in (0, 2):
            with pytest.raises(repro.ReproError):
                repro.repro_set_launch_cfg(fwd_selftest=v)
        repro.repro_set_launch_cfg(fwd_selftest=1)
        repro.repro_set_launch_cfg(fwd_path=2)
        repro.repro_set_launch_cfg(bwd_segment_log2=0, reduce_block_log2=0, fwd_path=0,
                                   elementwise_blocks=152)
    finally:
        repro.repro_set_launch_cfg(reset=True)


def test_optimiser_argument_checks(L):
    hp = repro.AdamWHparams(4.5e-4, 0.9, 0.95, 1e-8, 0.1, 1.0)
    f = L.repro_adamw_step
    B = 1 << 32
    assert f(B, B * 2, B * 3, B * 4, 100, B * 5, None, 1, None) == -1          # no hparams
    assert f(B, B * 2, B * 3, B * 4, 100, B * 5, ctypes.byref(hp), 0, None) == -1   # t < 1
    assert f(B, B * 2, B * 3, B * 4, -1, B * 5, ctypes.byref(hp), 1, None) == -2
    assert f(None, None, None, None, 0, None, ctypes.byref(hp), 1, None) == 0  # empty
    assert f(B + 4, B * 2, B * 3, B * 4, 100, B * 5, ctypes.byref(hp), 1, None) == -3
    assert f(B, B, B * 3, B * 4, 100, B * 5, ctypes.byref(hp), 1, None) == -8  # p is m
    assert L.repro_sumsq(B, 0, B * 2, B * 3, 1 << 20, None) == -2
    assert L.repro_sumsq(B, 1000, B * 2, None, 0, None) == -7
    assert L.repro_sumsq(None, 1000, B * 2, B * 3, 1 << 20, None) == -1
    assert repro.repro_sumsq_ws_bytes(10 ** 6) == repro.repro_wscale_ws_bytes(10 ** 6)


def test_running_sum_checks(L):
    P = ctypes.c_void_p
    parts = (P * 3)(A, A * 2, A * 3)
    assert L.repro_running_sum(parts, 0, 10, A * 4, None) == -1
    assert L.repro_running_sum(parts, 3, -1, A * 4, None) == -2
    assert L.repro_running_sum(parts, 3, 10, A * 3, None) == -8       # out overlaps parts[2]
    assert L.repro_running_sum(parts, 3, 0, A * 4, None) == 0


def test_launch_counter_readable(L):
    assert repro.repro_launch_count() >= 0


def test_state_hash_argument_checks(L):
    f = L.repro_state_hash
    P = ctypes.c_void_p
    I = ctypes.c_int64
    ptrs = lambda *v: (P * max(len(v), 1))(*v)          # noqa: E731
    sizes = lambda *v: (I * max(len(v), 1))(*v)         # noqa: E731
    D = A * 8   # digest
    W = A * 16  # workspace
    assert f(ptrs(A), sizes(10), -1, D, W, 1 << 20, None) == -1          # nbuf < 0
    assert f(ptrs(A), sizes(10), 65, D, W, 1 << 20, None) == -1          # nbuf > 64
    assert f(ptrs(A), sizes(10), 1, None, W, 1 << 20, None) == -1        # no digest
    assert f(None, None, 1, D, W, 1 << 20, None) == -1                   # no tables
    assert f(ptrs(A), sizes(-1), 1, D, W, 1 << 20, None) == -2           # negative size
    assert f(ptrs(None), sizes(10), 1, D, W, 1 << 20, None) == -1        # null buffer
    assert f(ptrs(A + 4), sizes(10), 1, D, W, 1 << 20, None) == -3       # misaligned buffer
    assert f(ptrs(A), sizes(10), 1, D + 8, W, 1 << 20, None) == -3       # misaligned digest
    big = 3 * 4096
    assert f(ptrs(A), sizes(big), 1, D, None, 0, None) == -7             # 3 leaves need ws
    assert f(ptrs(A), sizes(big), 1, D, W, 64, None) == -7               # too small
    assert f(ptrs(A), sizes(big), 1, W + 32, W, 1 << 20, None) == -8     # digest inside ws
    assert f(ptrs(W), sizes(big), 1, D, W, 1 << 20, None) == -8          # ws over a buffer
    # valid arguments reach the architecture check (no GPU here)
    assert f(ptrs(None), sizes(0), 1, D, None, 0, None) in (-4, -5)      # empty state
    assert f(ptrs(A), sizes(10), 1, D, None, 0, None) in (-4, -5)        # one leaf: no ws


def test_state_hash_ws_bytes(L):
    I = ctypes.c_int64
    g = L.repro_state_hash_ws_bytes
    assert g((I * 1)(0), 1) == 0
    assert g((I * 1)(4096), 1) == 0                     # one leaf: straight into the digest
    assert g((I * 2)(4096, 1), 2) == 256 + 256          # two leaves, one parent
    n = 1000 * 4096 + 5                                   # 1001 leaves + 501 parents
    assert g((I * 1)(n), 1) == ((1001 * 32 + 255) // 256) * 256 + ((501 * 32 + 255) // 256) * 256
    assert g((I * 1)(-1), 1) == 0


def test_attn_fwd_argument_checks(L):
    f = L.repro_attn_fwd
    Q, K, V, S, O, M, Lr = A, A * 2, A * 3, A * 4, A * 5, A * 6, A * 7
    args = lambda **k: [k.get("q", Q), k.get("k", K), k.get("vq", V), k.get("sv", S),   # noqa: E731
                        k.get("o", O), k.get("m", M), k.get("l", Lr), k.get("B", 1),
                        k.get("T", 8), k.get("Hq", 4), k.get("Hkv", 2), k.get("D", 128),
                        k.get("W", 0), k.get("ws", None), k.get("wsb", 0), None]
    assert f(*args(D=64)) == -2                      # head dim must be 128
    need = repro.repro_attn_fwd_ws_bytes(1, 8, 4, 0)
    # one query tile, one key tile, 4 heads: the logit cache, then the V^T and
    # K^T images of the tensor-core route (one 128 x 64 bf16 and one 128 x 64
    # fp32 tile per head, Hkv <= Hq)
    assert need == 4 * 64 * 64 * 4 + 4 * 128 * 64 * 2 + 4 * 128 * 64 * 4 + 16   # + work counter
    assert f(*args(ws=A * 16, wsb=need - 1)) == -7   # logit cache too small
    assert f(*args(ws=A * 16 + 8, wsb=need)) == -3   # misaligned cache
    assert f(*args(ws=Q, wsb=need)) == -8            # cache over q
    assert f(*args(Hkv=3)) == -2                     # Hq multiple of Hkv
    assert f(*args(T=131073)) == -2                  # exact int32 P.V bound
    assert f(*args(W=-1)) == -2
    assert f(*args(q=None)) == -1
    assert f(*args(o=O + 4)) == -3                   # misaligned
    assert f(*args(o=Q)) == -8                       # o over q
    assert f(*args(m=Lr)) == -8                      # m over l
    assert f(*args(B=0)) == 0                        # nothing to do
    assert f(*args()) in (-4, -5)                    # valid: reaches the architecture check


def test_attn_bwd_argument_checks(L):
    f = L.repro_attn_bwd
    names = ["q", "k", "vq", "sv", "o", "dout", "m", "l", "dq", "dk", "dv"]
    base = {n: A * (i + 1) for i, n in enumerate(names)}
    W_ = A * 32

    def args(**kw):
        v = dict(base, **{k: kw[k] for k in kw if k in base})
        return [v[n] for n in names] + [kw.get("B", 1), kw.get("T", 8), kw.get("Hq", 4),
                                        kw.get("Hkv", 2), kw.get("D", 128), kw.get("W", 0),
                                        kw.get("ws", W_), kw.get("wsb", 1 << 24),
                                        kw.get("fws", None), kw.get("fwsb", 0), None]
    assert f(*args(D=96)) == -2
    assert f(*args(Hkv=3)) == -2
    assert f(*args(dq=None)) == -1
    assert f(*args(dk=A * 2 + 4)) == -3
    assert f(*args(dq=A)) == -8                           # dq over q
    assert f(*args(dv=A * 10)) == -8                      # dv over dk
    assert f(*args(ws=None, wsb=0)) == -7
    assert f(*args(wsb=16)) == -7
    assert f(*args(ws=A)) == -8                           # ws over q
    assert f(*args(B=0)) == 0
    assert f(*args()) in (-4, -5)
    assert f(*args(fws=A * 64, fwsb=16)) == -7            # logit cache too small
    assert f(*args(fws=W_, fwsb=1 << 20)) == -8           # logit cache over ws
    # without the forward's cache: the int64 dQ accumulator and Dr_i
    assert repro.repro_attn_bwd_ws_bytes(1, 8, 4, -1) == 8 * 4 * 128 * 8 + 8 * 4 * 4
    # with it (one query tile, one key tile, 4 heads): also the a and dS tiles
    # (64 x 68 floats) and four 64 x 128-float images per head, 256-byte aligned
    need = repro.repro_attn_bwd_ws_bytes(1, 8, 4, 0)
    assert need >= 8 * 4 * 128 * 8 + 8 * 4 * 4 + 2 * 4 * 64 * 68 * 4 + 4 * 4 * 64 * 128 * 4 + 64
    assert need == repro.repro_attn_bwd_ws_bytes(1, 8, 4, 100)   # one tile either way


def test_selftest_arguments(L):
    need = L.repro_selftest_ws_bytes()
    assert need >= 128 * 1024 * 2 + 2 * 128 * 128 * 4
    assert L.repro_selftest(None, 0, None) == -7
    assert L.repro_selftest(A, need - 1, None) == -7
    assert L.repro_selftest(A + 4, need, None) == -3
    assert L.repro_selftest(A, need, None) in (-4, -5)   # valid: reaches the architecture check


def test_wait_probe_arguments(L):
    assert L.repro_wait_probe(2, None) == -1
    assert L.repro_wait_probe(-1, None) == -1
    assert L.repro_wait_probe(0, None) in (-4, -5)   # valid: reaches the architecture check
