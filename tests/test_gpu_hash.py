"""GPU parity of the on-device state hash (repro_state_hash, through the C ABI)
against the oracle's RFC 6962 Merkle Tree Hash over hashlib SHA-256: digests
must be byte-identical."""
import numpy as np
import pytest
import torch

import bitwise_reproducible_int8_gb300 as R

pytestmark = pytest.mark.gpu

LEAF = 4096


def _gpu_hash(arrays, stream=None):
    bufs = [torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).cuda()
            for a in arrays]
    digest = torch.zeros(32, dtype=torch.uint8, device="cuda")
    R.repro_state_hash(bufs, digest, stream=stream)
    torch.cuda.synchronize()
    assert R.repro_device_check() == 0
    return bytes(digest.cpu().numpy())


def _bytes(rng, n):
    return rng.integers(0, 256, n, dtype=np.uint8)


SIZES = [[], [0], [1], [2], [15], [63], [64], [65], [127], [4094], [LEAF - 1], [LEAF],
         [LEAF + 1], [2 * LEAF], [3 * LEAF + 17], [LEAF * 7 - 3], [5, 0, 3 * LEAF, 100],
         [0, 0], [LEAF, LEAF, 1], list(range(1, 40))]


@pytest.mark.parametrize("sizes", SIZES, ids=lambda s: "x".join(map(str, s)) or "none")
def test_state_hash_matches_oracle(orc, sizes):
    rng = np.random.default_rng(len(sizes) * 1000 + sum(sizes))
    arrays = [_bytes(rng, n) for n in sizes]
    assert _gpu_hash(arrays) == orc.state_hash([a.tobytes() for a in arrays])


@pytest.mark.parametrize("nleaves", [2, 3, 5, 8, 9, 33, 64, 65, 1000, 4097])
def test_tree_shapes(orc, nleaves):
    rng = np.random.default_rng(nleaves)
    a = _bytes(rng, nleaves * LEAF - (nleaves % 7))
    assert _gpu_hash([a]) == orc.state_hash([a.tobytes()])


def test_float_state_at_size(orc):
    # an optimiser state shaped like the block workload's: parameters and two
    # moment buffers of 45,088,768 fp32 values each (541 MB)
    rng = np.random.default_rng(42)
    n = 45088768
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = (rng.random(n) * 1e-8).astype(np.float32)
    assert _gpu_hash([p, m, v]) == orc.state_hash([p.tobytes(), m.tobytes(), v.tobytes()])


def test_one_flipped_bit_changes_the_digest():
    rng = np.random.default_rng(3)
    a = _bytes(rng, 10 * LEAF + 9)
    h = _gpu_hash([a])
    for pos in (0, LEAF - 1, LEAF, 5 * LEAF + 100, a.size - 1):
        b = a.copy()
        b[pos] ^= 0x80
        assert _gpu_hash([b]) != h, pos


def test_repeatable_across_streams():
    rng = np.random.default_rng(5)
    a = _bytes(rng, 300 * LEAF + 1)
    s = torch.cuda.Stream()
    assert _gpu_hash([a]) == _gpu_hash([a], stream=s)


def test_bench_input_digest_is_the_seeded_inputs():
    # the digest bench.py records is the Merkle root of exactly the seeded
    # inputs the step reads, in its stated order, and the same on a rerun
    from oracle import merkle
    from bitwise_reproducible_int8_gb300 import inputs, step
    wl = inputs.WORKLOADS["tiny"]
    host = step.generate_host_inputs(wl)
    hp = step.HotPathStep(wl, host)
    got = hp.input_digest()
    L, J = len(wl.linears), wl.microbatches
    bufs = [np.concatenate([w.ravel() for w in host.W]).tobytes()]
    bufs += [a.tobytes() for j in range(J) for i in range(L) for a in (host.X[i][j], host.dY[i][j])]
    assert got == merkle.state_hash(bufs).hex()
    assert step.HotPathStep(wl, step.generate_host_inputs(wl)).input_digest() == got
