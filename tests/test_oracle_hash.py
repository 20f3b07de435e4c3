"""Pins of the state-hash oracle (oracle/merkle.py) against things other
than itself: the published SHA-256 example vectors, an independent
level-by-level construction of the Merkle tree, the RFC 6962 / RFC 9162
inclusion-proof verification procedure, and the leaf-cutting rules."""
import hashlib
import random

import pytest

import oracle
from oracle import merkle as SH
from golden_io import sha256_vectors


def test_sha256_published_vectors():
    n = 0
    for msg, dig in sha256_vectors():
        assert SH.sha256(msg) == dig, msg
        n += 1
    assert n == 4


def _levels_root(data):
    # pair adjacent nodes level by level, carrying an odd last node up unchanged
    if not data:
        return hashlib.sha256(b"").digest()
    level = [hashlib.sha256(b"\x00" + d).digest() for d in data]
    while len(level) > 1:
        nxt = []
        for j in range(0, len(level) - 1, 2):
            nxt.append(hashlib.sha256(b"\x01" + level[j] + level[j + 1]).digest())
        if len(level) % 2:
            nxt.append(level[-1])
        level = nxt
    return level[0]


@pytest.mark.parametrize("n", list(range(0, 70)) + [127, 128, 129, 255, 256, 257])
def test_mth_equals_levelwise_pairing(n):
    rng = random.Random(n)
    data = [bytes(rng.getrandbits(8) for _ in range(rng.randrange(0, 9))) for _ in range(n)]
    assert SH.mth(data) == _levels_root(data)


def _verify_inclusion(m, n, leaf, path, root):
    # RFC 9162 section 2.1.3.2: walk the path with fn = m, sn = n - 1
    fn, sn = m, n - 1
    r = hashlib.sha256(b"\x00" + leaf).digest()
    for p in path:
        if sn == 0:
            return False
        if fn & 1 or fn == sn:
            r = hashlib.sha256(b"\x01" + p + r).digest()
            if not fn & 1:
                while fn and not fn & 1:
                    fn >>= 1
                    sn >>= 1
        else:
            r = hashlib.sha256(b"\x01" + r + p).digest()
        fn >>= 1
        sn >>= 1
    return sn == 0 and r == root


@pytest.mark.parametrize("n", [1, 2, 3, 5, 7, 8, 13, 31, 33])
def test_audit_paths_verify(n):
    rng = random.Random(100 + n)
    data = [bytes(rng.getrandbits(8) for _ in range(5)) for _ in range(n)]
    root = SH.mth(data)
    for m in range(n):
        assert _verify_inclusion(m, n, data[m], SH.audit_path(m, data), root)
    if n > 1:   # a wrong leaf or a wrong index fails
        assert not _verify_inclusion(0, n, data[0] + b"x", SH.audit_path(0, data), root)
        assert not _verify_inclusion(1, n, data[0], SH.audit_path(0, data), root)


def test_leaf_cutting():
    L = SH.LEAF_BYTES
    assert SH.leaves([b""]) == []
    assert SH.leaves([bytes(L)]) == [bytes(L)]
    assert [len(x) for x in SH.leaves([bytes(L + 1)])] == [L, 1]
    assert [len(x) for x in SH.leaves([bytes(3), bytes(2 * L)])] == [3, L, L]
    # empty state: the hash of the empty string; one empty buffer is the same
    assert SH.state_hash([]) == hashlib.sha256(b"").digest()
    assert SH.state_hash([b"", b""]) == SH.state_hash([])
    # one short buffer: the leaf hash of its bytes
    assert SH.state_hash([b"abc"]) == hashlib.sha256(b"\x00abc").digest()


def test_splitting_at_a_leaf_boundary_keeps_the_hash_and_elsewhere_changes_it():
    rng = random.Random(7)
    L = 64
    buf = bytes(rng.getrandbits(8) for _ in range(5 * L + 17))
    h = SH.state_hash([buf], leaf_bytes=L)
    assert SH.state_hash([buf[:2 * L], buf[2 * L:]], leaf_bytes=L) == h
    assert SH.state_hash([buf[:2 * L + 1], buf[2 * L + 1:]], leaf_bytes=L) != h


def test_every_byte_and_the_leaf_order_matter():
    rng = random.Random(11)
    L = 32
    buf = bytearray(rng.getrandbits(8) for _ in range(7 * L + 5))
    h = SH.state_hash([bytes(buf)], leaf_bytes=L)
    for pos in (0, 1, L - 1, L, 3 * L + 7, len(buf) - 1):
        b2 = bytearray(buf)
        b2[pos] ^= 0x01
        assert SH.state_hash([bytes(b2)], leaf_bytes=L) != h, pos
    lv = SH.leaves([bytes(buf)], L)
    lv[1], lv[2] = lv[2], lv[1]
    assert SH.mth(lv) != h


def test_exported_from_package():
    assert oracle.state_hash is SH.state_hash
    assert oracle.HASH_LEAF_BYTES == 4096
