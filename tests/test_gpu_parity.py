"""GPU parity: every output of the C-ABI library against the CPU oracle,
element by element, bit for bit (0 ULP), on seeded inputs that span several
tiles and chunks with ragged tails, plus the edge cases of the method."""
import numpy as np
import pytest

from bitwise_reproducible_int8_gb300 import inputs
from golden_io import bits_to_f32, canon_cases, ftz_cases, quant_cases, treefold_cases

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import gpu_helpers as G  # noqa: E402
import bitwise_reproducible_int8_gb300 as R  # noqa: E402


@pytest.fixture(autouse=True)
def _default_cfg():
    R.repro_set_launch_cfg(reset=True)
    yield
    R.repro_set_launch_cfg(reset=True)


def _specials(rng, n):
    x = (rng.standard_normal(n) * 10.0 ** rng.integers(-3, 3, n)).astype(np.float32)
    k = min(n, 12)
    x[:k] = np.array([0.0, -0.0, 1e-40, -1e-40, 1.17549435e-38, -2.5, 2.5, 1e30, -1e30,
                      3e-39, 0.5, -0.5][:k], dtype=np.float32)
    rng.shuffle(x)
    return x


# ----------------------------------------------------------------- scales

@pytest.mark.parametrize("n", [1, 2, 63, 64, 65, 127, 129, 1000, 8191, 8192 + 64 * 3 + 5,
                               300_001, 1 << 20, (1 << 20) + 77])
@pytest.mark.parametrize("mode", [0, 1])
def test_scale(orc, n, mode):
    rng = np.random.default_rng(n * 2 + mode)
    x = _specials(rng, n) if n > 20 else (rng.standard_normal(n) * 0.02).astype(np.float32)
    G.assert_bits_equal(np.float32(G.gpu_scale(x, mode)), np.float32(orc.wscale(x, mode)),
                        f"scale mode {mode} n {n}")


def test_scale_discriminators(orc):
    # |x| of the canonical-order fixtures: the absolute values still discriminate
    for p, _ in canon_cases():
        if p.size == 0:
            continue
        G.assert_bits_equal(np.float32(G.gpu_scale(p, 0)), np.float32(orc.wscale(p, 0)),
                            f"scale discriminator L={p.size}")


@pytest.mark.parametrize("blk", [0, 1, 2, 3, 5, 7, 8, 10])
def test_scale_launch_invariance(orc, blk):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(700_003) * 0.02).astype(np.float32)
    ref = np.float32(orc.wscale(x, 0))
    R.repro_set_launch_cfg(reduce_block_log2=blk)
    G.assert_bits_equal(np.float32(G.gpu_scale(x, 0)), ref, f"block 2^{blk}")


@pytest.mark.parametrize("n", [1, 100, 700_003])
@pytest.mark.parametrize("grid", [1, 7, 152, 5000])
def test_amax_grid_invariance(orc, n, grid):
    # the launch-configuration hook sets the amax grid (capped by the
    # workspace's partial slots); the maximum is exact whatever the split
    rng = np.random.default_rng(n + grid)
    x = rng.standard_normal(n).astype(np.float32)
    ref = np.float32(orc.wscale(x, 1))
    R.repro_set_launch_cfg(elementwise_blocks=grid)
    G.assert_bits_equal(np.float32(G.gpu_scale(x, 1)), ref, f"amax n {n} grid {grid}")


def test_scale_non_finite(orc):
    # the activation scale's maximum passes over NaN elements and an infinite
    # one makes it infinite; the weight scale's sum carries a NaN (any NaN
    # pattern) and an infinity through
    rng = np.random.default_rng(8)
    base = rng.standard_normal(70_000).astype(np.float32)
    for bad in (np.nan, np.inf, -np.inf):
        x = base.copy()
        x[[3, 4097, 69_999]] = bad
        for mode in (0, 1):
            got, exp = np.float32(G.gpu_scale(x, mode)), np.float32(orc.wscale(x, mode))
            if np.isnan(exp):
                assert np.isnan(got), (bad, mode)
            else:
                G.assert_bits_equal(got, exp, f"scale mode {mode} with {bad}")
        if np.isnan(bad):
            assert np.isfinite(orc.wscale(x, 1))


# ----------------------------------------------------------------- quantiser

@pytest.mark.parametrize("n", [1, 15, 16, 17, 1000, 65536 + 9])
def test_quant(orc, n):
    rng = np.random.default_rng(n)
    x = _specials(rng, n) if n > 20 else rng.standard_normal(n).astype(np.float32)
    for s in [np.float32(0.0284), np.float32(1.0), np.float32(3e-3)]:
        G.assert_bits_equal(G.gpu_quant(x, s), orc.quant_i8(x, s), f"quant n {n} s {s}")


def test_quant_golden(orc):
    for xb, sb, q in quant_cases():
        x = np.array([bits_to_f32(xb)], dtype=np.float32)
        got = G.gpu_quant(x, bits_to_f32(sb))
        assert int(got[0]) == q, (hex(xb), hex(sb), int(got[0]))


def test_quant_non_finite(orc):
    # a NaN quotient gives 0 and infinite ones clamp to +-127, as the oracle
    # states; the 16-element groups of the kernel and its ragged tail both
    x = np.array([np.nan, np.inf, -np.inf, 1.0, -np.nan, 3.0e38, -3.0e38, 0.5], np.float32)
    x = np.concatenate([x, x[::-1], x[:5]])
    for s in [np.float32(0.0284), np.float32(1.0), np.float32(1e-30)]:
        exp = orc.quant_i8(x, s)
        assert list(exp[:3]) == [0, 127, -127]
        G.assert_bits_equal(G.gpu_quant(x, s), exp, f"non-finite quotients, s {s}")


def test_quant_half_integers(orc):
    s = np.float32(0.0371)
    x = ((np.arange(-300, 300, dtype=np.float32) + np.float32(0.5)) * s).astype(np.float32)
    G.assert_bits_equal(G.gpu_quant(x, s), orc.quant_i8(x, s), "half-integer quotients")


# ----------------------------------------------------------------- forward

FWD_SHAPES = [(1, 1, 1), (3, 5, 7), (64, 128, 256), (130, 70, 200), (65, 129, 1040),
              (200, 96, 2048), (17, 300, 33), (257, 129, 5632), (128, 128, 8), (300, 260, 520),
              (130, 384, 1024), (200, 500, 1536), (129, 514, 1032), (256, 512, 4096)]


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", FWD_SHAPES)
def test_forward(orc, M, N, K, path):
    R.repro_set_launch_cfg(fwd_path=path)
    rng = np.random.default_rng(M + N + K)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    s_x, s_w = np.float32(0.0371), np.float32(0.00284)
    G.assert_bits_equal(G.gpu_fwd(xq, wq, s_x, s_w), orc.linear_fwd(xq, wq, s_x, s_w),
                        f"fwd {M}x{N}x{K}")


# more output tiles than SMs, so the persistent tensor-core forward walks
# several tiles per CTA and its K-slice counters and accumulator buffers carry
# across tiles: ragged rows and columns, row pitches with and without 16-byte
# multiples (TMA-store and register-store epilogues), one to three K-slices
FWD_MULTI_TILE = [(1300, 4100, 1096), (1300, 4099, 1096), (2177, 2052, 520), (4096, 4096, 64)]


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", FWD_MULTI_TILE)
def test_forward_many_tiles_per_cta(orc, M, N, K, path):
    R.repro_set_launch_cfg(fwd_path=path)
    rng = np.random.default_rng(M * 7 + N + K)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    s_x, s_w = np.float32(0.0213), np.float32(0.00391)
    want = orc.linear_fwd(xq, wq, s_x, s_w)
    for _ in range(2):   # and the same bits on a second call
        G.assert_bits_equal(G.gpu_fwd(xq, wq, s_x, s_w), want, f"fwd {M}x{N}x{K} path {path}")


def test_tensor_core_forward_selftest():
    # adversarial codes through the tensor-core path and the exact dp4a path
    assert R.repro_selftest() == R.REPRO_OK


def _fwd_launches(xq, wq, s_x, s_w):
    torch.cuda.synchronize()
    before = R.repro_launch_count()
    y = G.gpu_fwd(xq, wq, s_x, s_w)
    return y, R.repro_launch_count() - before


def test_forward_gate_takes_the_tensor_cores_after_a_passed_check(orc):
    # default path: the device's exactness check has passed (it runs on the
    # first tensor-core call; every later call goes straight to the tensor
    # cores: two int8 -> bf16 widening passes and the tensor-core kernel)
    rng = np.random.default_rng(5)
    xq = rng.integers(-127, 128, (300, 1024)).astype(np.int8)
    wq = rng.integers(-127, 128, (260, 1024)).astype(np.int8)
    s_x, s_w = np.float32(0.0371), np.float32(0.00284)
    G.gpu_fwd(xq, wq, s_x, s_w)
    assert R.repro_device_check() == R.REPRO_OK        # no failed check to report
    y, n = _fwd_launches(xq, wq, s_x, s_w)
    G.assert_bits_equal(y, orc.linear_fwd(xq, wq, s_x, s_w), "gated forward")
    assert n == 3, n


def test_forward_gate_falls_back_to_the_exact_path(orc):
    # the test hook acts as if the check had failed: the same call takes the
    # CUDA-core (dp4a) kernel alone, gives the oracle's bits, and the next
    # device check reports the failure once
    R.repro_set_launch_cfg(fwd_selftest=1)
    rng = np.random.default_rng(6)
    xq = rng.integers(-127, 128, (300, 1024)).astype(np.int8)
    wq = rng.integers(-127, 128, (260, 1024)).astype(np.int8)
    s_x, s_w = np.float32(0.0371), np.float32(0.00284)
    y, n = _fwd_launches(xq, wq, s_x, s_w)
    G.assert_bits_equal(y, orc.linear_fwd(xq, wq, s_x, s_w), "fallback forward")
    assert n == 1, n
    assert R.repro_device_check() == -9                 # REPRO_ERR_SELFTEST
    assert R.repro_device_check() == R.REPRO_OK
    R.repro_set_launch_cfg(reset=True)
    y, n = _fwd_launches(xq, wq, s_x, s_w)
    assert n == 3 and R.repro_device_check() == R.REPRO_OK


@pytest.mark.parametrize("path", [0, 1, 2])
def test_forward_at_the_maximum_reduction(orc, path):
    # K = 133,144 is the largest K for which |acc| <= 127 * 127 * K fits int32;
    # codes at the clamp make row 0 reach 2,147,479,576
    R.repro_set_launch_cfg(fwd_path=path)
    K = 133144
    rng = np.random.default_rng(5)
    xq = rng.integers(-127, 128, (5, K)).astype(np.int8)
    wq = rng.integers(-127, 128, (7, K)).astype(np.int8)
    xq[0] = 127
    wq[0] = 127
    wq[1] = -127
    y = G.gpu_fwd(xq, wq, np.float32(1.0), np.float32(1.0))
    G.assert_bits_equal(y, orc.linear_fwd(xq, wq, 1.0, 1.0), "fwd K max")
    assert orc.int_dot(xq, wq, 0, 0) == 127 * 127 * K


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("K", [1024, 1040, 2048, 5632])
def test_forward_adversarial(orc, K, path):
    R.repro_set_launch_cfg(fwd_path=path)
    # all codes at the clamp: |acc| = 16129 K, above 2^24 for K > 1040
    M, N = 4, 4
    xq = np.full((M, K), 127, np.int8)
    xq[1] = -127
    xq[2, ::2] = -127
    xq[3, ::3] = 0
    wq = np.full((N, K), 127, np.int8)
    wq[1] = -127
    wq[2, 1::2] = -127
    wq[3, ::5] = 1
    G.assert_bits_equal(G.gpu_fwd(xq, wq, np.float32(1.0), np.float32(1.0)),
                        orc.linear_fwd(xq, wq, 1.0, 1.0), f"fwd adversarial K={K}")


# ----------------------------------------------------------------- backward

# the two shipped backward kernels: 8 (default, tensor-copy fed, 16-byte-aligned
# rows) and 1 (register prefetch, any rows); unaligned shapes run 1 either way
BWD_KERNELS = [1, 8]

BWD_SHAPES = [(1, 1, 1), (3, 1, 5), (64, 128, 256), (200, 130, 70), (257, 64, 65),
              (130, 257, 96), (64, 64, 64), (1000, 300, 17), (96, 4100, 20),
              (257, 68, 96), (100, 4100, 32), (1000, 300, 16), (70, 132, 48), (300, 260, 80)]


@pytest.mark.parametrize("kernel", BWD_KERNELS)
@pytest.mark.parametrize("M,N,K", BWD_SHAPES)
def test_backward(orc, M, N, K, kernel):
    R.repro_set_launch_cfg(bwd_kernel=kernel)
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    s_x, s_w = np.float32(0.0311), np.float32(0.00277)
    dx, dw = G.gpu_bwd(dy, xq, wq, s_x, s_w)
    G.assert_bits_equal(dx, orc.linear_bwd_dx(dy, wq, s_w), f"dx {M}x{N}x{K}")
    G.assert_bits_equal(dw, orc.linear_bwd_dw(dy, xq, s_x), f"dw {M}x{N}x{K}")


@pytest.mark.parametrize("kernel", BWD_KERNELS)
@pytest.mark.parametrize("seg", [0, 1, 2, 3, 4, 8])
def test_backward_launch_invariance(orc, seg, kernel):
    # long reductions split into aligned segments of 2^seg chunks, by either kernel
    rng = np.random.default_rng(seg)
    M, N, K = 1100, 900, 48
    dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    R.repro_set_launch_cfg(bwd_segment_log2=seg, bwd_kernel=kernel)
    dx, dw = G.gpu_bwd(dy, xq, wq, np.float32(0.03), np.float32(0.003))
    G.assert_bits_equal(dx, orc.linear_bwd_dx(dy, wq, np.float32(0.003)), f"dx seg {seg}")
    G.assert_bits_equal(dw, orc.linear_bwd_dw(dy, xq, np.float32(0.03)), f"dw seg {seg}")


def test_backward_long_reduction(orc):
    # dW over 70,000 tokens: 1094 chunks, more than one 256-chunk segment at the
    # default launch, so the segment partials meet in the pairwise passes
    rng = np.random.default_rng(70000)
    M, N, K = 70000, 8, 32
    dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    _, dw = G.gpu_bwd(dy, xq, None, np.float32(0.031), None, want_dx=False)
    G.assert_bits_equal(dw, orc.linear_bwd_dw(dy, xq, np.float32(0.031)), "dw M=70000")


def test_backward_discriminators(orc):
    # route each canonical-order fixture through dX and dW: products equal the
    # fixture's terms (scale 1, codes 1), so chunking, order and tree shape all
    # show in the bits
    for p, exp in canon_cases():
        L = p.size
        if L == 0:
            continue
        dy = np.zeros((2, L), np.float32)
        dy[1] = p
        wq = np.ones((L, 3), np.int8)
        dx, _ = G.gpu_bwd(dy, None, wq, None, np.float32(1.0), want_dw=False)
        assert int(dx[1, 1:2].view(np.uint32)[0]) == exp, (L, hex(exp))
        dyt = np.ascontiguousarray(dy.T)            # [L, 2]
        xq = np.ones((L, 3), np.int8)
        _, dw = G.gpu_bwd(dyt, xq, None, np.float32(1.0), None, want_dx=False)
        assert int(dw[1, 2:3].view(np.uint32)[0]) == exp, (L, hex(exp))


def test_backward_flush_cases(orc):
    # products that land below FLT_MIN, on it, and subnormal upstream gradients
    M, N, K = 3, 70, 2
    dy = np.full((M, N), 1.1754944e-38, np.float32)      # FLT_MIN
    dy[1] = 1e-40                                        # subnormal: read as 0
    dy[2, ::2] = -3.0e-38
    wq = np.ones((N, K), np.int8)
    wq[:, 1] = 127
    for s_w in [np.float32(0.5), np.float32(0.99999994), np.float32(1.0)]:
        dx, _ = G.gpu_bwd(dy, None, wq, None, s_w, want_dw=False)
        G.assert_bits_equal(dx, orc.linear_bwd_dx(dy, wq, s_w), f"flush s_w={s_w}")


@pytest.mark.parametrize("kernel", BWD_KERNELS)
def test_backward_subnormal_dy_every_kernel(orc, kernel):
    # subnormal upstream gradients against codes of 127 at scale 1: unflushed,
    # 1e-40 (x) 127 = 1.27e-38 would be a normal product, so a missed flush of
    # dY changes dX and dW; the shape is aligned, so kernel 8 takes its
    # fast paths (dW over 130 tokens: three chunks, a ragged tail)
    R.repro_set_launch_cfg(bwd_kernel=kernel)
    rng = np.random.default_rng(40)
    M, N, K = 130, 68, 32
    dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    dy[::3, ::2] = 1e-40
    dy[1::5, 1::3] = -1e-40
    dy[7] = 1e-40                                         # a whole row
    dy[:, 5] = -1e-40                                     # a whole column
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    xq[::2] = 127
    wq[::2] = -127
    one = np.float32(1.0)
    dx, dw = G.gpu_bwd(dy, xq, wq, one, one)
    G.assert_bits_equal(dx, orc.linear_bwd_dx(dy, wq, one), f"dx kernel {kernel}")
    G.assert_bits_equal(dw, orc.linear_bwd_dw(dy, xq, one), f"dw kernel {kernel}")


def test_backward_accumulate_flag(orc):
    rng = np.random.default_rng(21)
    M, N, K = 300, 130, 68
    dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    acc0 = (rng.standard_normal((N, K)) * 1e-2).astype(np.float32)
    acc0[0, :4] = [-0.0, 0.0, 1e-40, -1e-40]
    dwt = G.dev(acc0.copy())
    R.repro_linear_bwd(G.dev(dy), G.dev(xq), None, G.scalar(0.03), None, None, dwt,
                       accumulate=True)
    ref = orc.grad_accum(acc0, orc.linear_bwd_dw(dy, xq, np.float32(0.03)))
    G.assert_bits_equal(G.host(dwt), ref, "fused accumulate")


def test_backward_empty_reduction(orc):
    # N = 0: dX is the empty canonical sum, +0 everywhere
    dx = torch.full((4, 8), 7.0, device="cuda")
    R.repro_linear_bwd(torch.empty((4, 0), device="cuda"), None,
                       torch.empty((0, 8), dtype=torch.int8, device="cuda"), None,
                       G.scalar(1.0), dx, None)
    assert np.all(G.host(dx).view(np.uint32) == 0)


@pytest.mark.parametrize("kernel", BWD_KERNELS)
def test_zero_weights_and_activations_every_kernel(orc, kernel):
    # all-zero W and X: both scales are +0, every code is 0, and every
    # backward product is a signed zero, so the sign of each dX and dW element
    # comes from the seeded chunk sums and the pairwise tree alone
    # (+0 (+) -0 = +0, -0 (+) -0 = -0); rows and columns of dY that are
    # entirely negative give -0 results, mixed ones +0
    R.repro_set_launch_cfg(bwd_kernel=kernel)
    rng = np.random.default_rng(41)
    M, N, K = 130, 136, 32
    w = np.zeros((N, K), np.float32)
    x = np.zeros((M, K), np.float32)
    x[3, :4] = -0.0
    s_w = G.gpu_scale(w, 0)
    s_x = G.gpu_scale(x, 1)
    G.assert_bits_equal(np.float32(s_w), orc.wscale(w, 0), "s_w of zeros")
    G.assert_bits_equal(np.float32(s_x), orc.wscale(x, 1), "s_x of zeros")
    wq, xq = G.gpu_quant(w, s_w), G.gpu_quant(x, s_x)
    assert not wq.any() and not xq.any()
    dy = np.abs(rng.standard_normal((M, N))).astype(np.float32) * 1e-3
    dy[::2] *= -1                                   # whole negative rows
    dy[:, 7] = -np.abs(dy[:, 7])                    # a whole negative column
    dy[5, :70] = -1e-3                              # negative across the first chunk only
    G.assert_bits_equal(G.gpu_fwd(xq, wq, s_x, s_w), orc.linear_fwd(xq, wq, s_x, s_w), "fwd 0")
    dx, dw = G.gpu_bwd(dy, xq, wq, s_x, s_w)
    G.assert_bits_equal(dx, orc.linear_bwd_dx(dy, wq, s_w), f"dx of zero weights, kernel {kernel}")
    G.assert_bits_equal(dw, orc.linear_bwd_dw(dy, xq, s_x), f"dw of zero activations, kernel {kernel}")
    assert (dx.view(np.uint32) == 0x80000000).any() and (dx.view(np.uint32) == 0).any()


# ----------------------------------------------------------------- reductions

@pytest.mark.parametrize("n", [1, 3, 4, 5, 1000, 65536 + 3])
def test_grad_accum(orc, n):
    rng = np.random.default_rng(n)
    a = _specials(rng, n) if n > 20 else rng.standard_normal(n).astype(np.float32)
    g = _specials(rng, n) if n > 20 else rng.standard_normal(n).astype(np.float32)
    G.assert_bits_equal(G.gpu_accum(a, g), orc.grad_accum(a, g), f"accum n {n}")


@pytest.mark.parametrize("R_", [1, 2, 3, 4, 5, 6, 7, 8, 9, 13, 16, 33, 64])
def test_treefold(orc, R_):
    rng = np.random.default_rng(R_)
    n = 4099
    parts = [(rng.standard_normal(n) * 10.0 ** rng.integers(-3, 3, n)).astype(np.float32)
             for _ in range(R_)]
    parts[0][:4] = [1e-40, -0.0, 2.0 ** 24, -1e-40]
    G.assert_bits_equal(G.gpu_treefold(parts), orc.treefold(parts), f"treefold R={R_}")


def test_treefold_golden():
    for vals, exp in treefold_cases():
        parts = [np.array([v] * 5, dtype=np.float32) for v in vals]
        got = G.gpu_treefold(parts)
        assert np.all(got.view(np.uint32) == exp), (vals, hex(exp))


def test_treefold_in_place_and_layout(orc):
    rng = np.random.default_rng(8)
    Rn, n = 6, 10_004          # rows of the block stay 16-byte aligned
    block = (rng.standard_normal((Rn, n)) * 1e-3).astype(np.float32)
    ref = orc.treefold([block[r] for r in range(Rn)])
    tb = G.dev(block)
    views = [tb[r] for r in range(Rn)]
    out = torch.empty(n, device="cuda")
    R.repro_treefold(views, out)
    G.assert_bits_equal(G.host(out), ref, "contiguous block")
    rev = G.dev(np.ascontiguousarray(block[::-1]))
    R.repro_treefold([rev[Rn - 1 - r] for r in range(Rn)], out)
    G.assert_bits_equal(G.host(out), ref, "reversed memory order")
    sep = [G.dev(block[r].copy()) for r in range(Rn)]
    R.repro_treefold(sep, sep[0])                       # out aliases parts[0]
    G.assert_bits_equal(G.host(sep[0]), ref, "in place")


def test_ftz_cases_through_kernels(orc):
    # the elementary flush cases, evaluated by the GPU's add (grad_accum) and
    # multiply (one-term backward: dX = dY (x) (1 (x) s_w))
    for op, a, b, exp in ftz_cases():
        fa = np.array([bits_to_f32(a)] * 4, np.float32)
        fb = np.array([bits_to_f32(b)] * 4, np.float32)
        if op == "add":
            got = G.gpu_accum(fa, fb)
            assert np.all(got.view(np.uint32) == exp), (op, hex(a), hex(b))
        elif op == "mul":
            dy = fa.reshape(4, 1)
            wq = np.ones((1, 1), np.int8)
            dx, _ = G.gpu_bwd(dy, None, wq, None, fb[0], want_dw=False)
            G.assert_bits_equal(dx, orc.linear_bwd_dx(dy, wq, fb[0]), f"mul {a:08x} {b:08x}")


# ----------------------------------------------------------------- tiny workload end to end

def test_tiny_workload_end_to_end(orc):
    wl = inputs.WORKLOADS["tiny"]
    X = inputs.activation(wl, 0, 0)
    W = inputs.weight(wl, 0)
    dY = inputs.upstream_grad(wl, 0, 0)
    # oracle side
    s_w = orc.wscale(W, 0)
    s_x = orc.wscale(X, 1)
    wq, xq = orc.quant_i8(W, s_w), orc.quant_i8(X, s_x)
    y = orc.linear_fwd(xq, wq, s_x, s_w)
    dx, dw = orc.linear_bwd_dx(dY, wq, s_w), orc.linear_bwd_dw(dY, xq, s_x)
    noise = [inputs.replica_noise(wl, r, dw.size).reshape(dw.shape) for r in range(wl.replicas)]
    reps = [orc.grad_accum(dw, nz) for nz in noise]
    tf = orc.treefold(reps).reshape(dw.shape)
    # GPU side, same host inputs
    Wt, Xt, dYt = G.dev(W), G.dev(X), G.dev(dY)
    sw_t, sx_t = torch.empty(1, device="cuda"), torch.empty(1, device="cuda")
    R.repro_wscale(Wt, 0, sw_t)
    R.repro_wscale(Xt, 1, sx_t)
    wq_t = torch.empty(W.shape, dtype=torch.int8, device="cuda")
    xq_t = torch.empty(X.shape, dtype=torch.int8, device="cuda")
    R.repro_quant_i8(Wt, sw_t, wq_t)
    R.repro_quant_i8(Xt, sx_t, xq_t)
    y_t = torch.empty(y.shape, device="cuda")
    R.repro_linear_fwd(xq_t, wq_t, sx_t, sw_t, y_t)
    dx_t, dw_t = torch.empty(dx.shape, device="cuda"), torch.empty(dw.shape, device="cuda")
    R.repro_linear_bwd(dYt, xq_t, wq_t, sx_t, sw_t, dx_t, dw_t)
    reps_t = []
    for nz in noise:
        r = dw_t.clone()
        R.repro_grad_accum(r, G.dev(nz))
        reps_t.append(r)
    tf_t = torch.empty_like(dw_t)
    R.repro_treefold(reps_t, tf_t)
    for name, got, exp in [("s_w", G.host(sw_t), np.float32([s_w])),
                           ("s_x", G.host(sx_t), np.float32([s_x])),
                           ("Wq", G.host(wq_t), wq), ("Xq", G.host(xq_t), xq),
                           ("Y", G.host(y_t), y), ("dX", G.host(dx_t), dx),
                           ("dW", G.host(dw_t), dw), ("TreeFold", G.host(tf_t), tf)]:
        G.assert_bits_equal(got, exp, name)


# ----------------------------------------------------------------- level 2

@pytest.mark.parametrize("S_", [1, 2, 3, 5, 8, 9, 16, 64])
def test_running_sum(orc, S_):
    rng = np.random.default_rng(300 + S_)
    n = 4099
    parts = [(rng.standard_normal(n) * 10.0 ** rng.integers(-3, 3, n)).astype(np.float32)
             for _ in range(S_)]
    parts[0][:4] = [1e-40, -0.0, 2.0 ** 24, -1e-40]
    ts = [G.dev(p) for p in parts]
    out = torch.empty_like(ts[0])
    R.repro_running_sum(ts, out)
    G.assert_bits_equal(G.host(out), orc.running_sum(parts), f"running sum S={S_}")
    R.repro_running_sum(ts, ts[0])                       # in place into the first partial
    G.assert_bits_equal(G.host(ts[0]), orc.running_sum(parts), f"running sum in place S={S_}")


def test_running_sum_equals_streaming_accumulation():
    rng = np.random.default_rng(7)
    parts = [G.dev((rng.standard_normal(10_000) * 1e-3).astype(np.float32)) for _ in range(8)]
    out = torch.empty_like(parts[0])
    R.repro_running_sum(parts, out)
    acc = parts[0].clone()
    for p in parts[1:]:
        R.repro_grad_accum(acc, p)
    G.assert_bits_equal(G.host(out), G.host(acc), "one pass vs streaming")


# ----------------------------------------------------------- several tensors

MULTI_SIZES = [[1], [5, 64, 65], [8192 * 3 + 17, 1000, 1, 16, 17], [300_001, 700_003, 63, 8192]]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("sizes", MULTI_SIZES, ids=lambda s: "x".join(map(str, s)))
def test_multi_tensor_scale_and_quant(orc, sizes, mode):
    # one call over several tensors: the oracle's bits for every tensor's
    # scale, then every tensor's codes with its own scale
    rng = np.random.default_rng(sum(sizes) + mode)
    xh = [_specials(rng, n) if n > 20 else (rng.standard_normal(n) * 0.02).astype(np.float32)
          for n in sizes]
    xs = [G.dev(x) for x in xh]
    scales = torch.full((len(sizes),), float("nan"), device="cuda")
    R.repro_wscale_multi(xs, mode, scales)
    got = G.host(scales)
    exp = np.array([orc.wscale(x, mode) for x in xh], dtype=np.float32)
    G.assert_bits_equal(got, exp, f"multi scale mode {mode}")
    qs = [torch.empty(n, dtype=torch.int8, device="cuda") for n in sizes]
    R.repro_quant_i8_multi(xs, scales, qs)
    for x, q, s in zip(xh, qs, exp):
        G.assert_bits_equal(G.host(q), orc.quant_i8(x, s), f"multi quant n {x.size}")


@pytest.mark.parametrize("blk", [0, 3, 7])
@pytest.mark.parametrize("grid", [0, 1, 5, 3000])
def test_multi_tensor_launch_invariance(orc, blk, grid):
    # block split (at 2^0 chunks per block the 700,003-element tensor needs
    # more partials than one tree CTA holds: every tensor then takes the
    # single-tensor passes) and the quantiser's grid, including fewer CTAs
    # than tensors
    sizes = [700_003, 100, 64 * 129, 17]
    rng = np.random.default_rng(blk * 10 + grid)
    xh = [(rng.standard_normal(n) * 0.02).astype(np.float32) for n in sizes]
    xs = [G.dev(x) for x in xh]
    exp = np.array([orc.wscale(x, 0) for x in xh], dtype=np.float32)
    R.repro_set_launch_cfg(reduce_block_log2=blk, elementwise_blocks=grid)
    scales = torch.empty(len(sizes), device="cuda")
    R.repro_wscale_multi(xs, 0, scales)
    G.assert_bits_equal(G.host(scales), exp, f"block 2^{blk}")
    qs = [torch.empty(n, dtype=torch.int8, device="cuda") for n in sizes]
    R.repro_quant_i8_multi(xs, scales, qs)
    for x, q, s in zip(xh, qs, exp):
        G.assert_bits_equal(G.host(q), orc.quant_i8(x, s), f"grid {grid} n {x.size}")
    # a zero scale gives zero codes, as in the single-tensor quantiser
    zs = torch.zeros(len(sizes), device="cuda")
    R.repro_quant_i8_multi(xs, zs, qs)
    for q in qs:
        assert not G.host(q).any()


@pytest.mark.parametrize("extra", [0, 1])
def test_multi_tensor_scale_at_the_one_pass_limit(orc, extra):
    # 8192 blocks of 8192 elements is the most one tree CTA takes; one element
    # more sends the call through the single-tensor passes: same bits either way
    n = 8192 * 8192 + extra
    rng = np.random.default_rng(81 + extra)
    xh = (rng.standard_normal(n) * 0.02).astype(np.float32)
    small = (rng.standard_normal(1000) * 0.02).astype(np.float32)
    scales = torch.empty(2, device="cuda")
    R.repro_wscale_multi([G.dev(xh), G.dev(small)], 0, scales)
    exp = np.array([orc.wscale(xh, 0), orc.wscale(small, 0)], dtype=np.float32)
    G.assert_bits_equal(G.host(scales), exp, f"n {n}")
