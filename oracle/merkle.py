"""Oracle of the per-step state hash (TEST INFRASTRUCTURE, like the rest of
``oracle/``: only tests, ``__graft_entry__.smoke()`` and the benchmark's CPU
legs may import it).

The pages record a hash of the training state after every optimiser step so
that a replay can be compared with the original run; they compute it on the
host and name on-device hashing as future work (Open-1B review,
onedev.kr/papers/92, section "Premises and limits"; rit.work blog
"open-1b-auditable-training", paragraph 4).  They do not fix the construction.
The reading taken here is the Merkle Tree Hash of RFC 6962 (Certificate
Transparency, section 2.1) over SHA-256 (FIPS 180-4):

  * the state is a list of byte buffers; each buffer is cut into leaves of
    LEAF_BYTES consecutive bytes (the last leaf of a buffer may be shorter, an
    empty buffer has no leaves); the leaf sequence is the buffers' leaves in
    buffer order;
  * MTH({}) = SHA-256(""),
    MTH({d}) = SHA-256(0x00 || d),
    MTH(D[0:n]) = SHA-256(0x01 || MTH(D[0:k]) || MTH(D[k:n])) for n > 1, with k
    the largest power of two smaller than n.

Written from the RFC's recursive definition; SHA-256 itself is the library
routine ``hashlib.sha256`` (pinned by the FIPS 180-2 example vectors in the
tests).
"""
from __future__ import annotations

import hashlib
from typing import Iterable, List, Sequence

LEAF_BYTES = 4096


def sha256(b: bytes) -> bytes:
    return hashlib.sha256(b).digest()


def leaves(buffers: Iterable[bytes], leaf_bytes: int = LEAF_BYTES) -> List[bytes]:
    """The leaf sequence: every buffer cut into leaf_bytes pieces, in order."""
    out: List[bytes] = []
    for buf in buffers:
        buf = bytes(buf)
        for off in range(0, len(buf), leaf_bytes):
            out.append(buf[off:off + leaf_bytes])
    return out


def mth(data: Sequence[bytes]) -> bytes:
    """RFC 6962 section 2.1 Merkle Tree Hash of a list of leaf inputs."""
    n = len(data)
    if n == 0:
        return sha256(b"")
    if n == 1:
        return sha256(b"\x00" + data[0])
    k = 1
    while k * 2 < n:
        k *= 2
    return sha256(b"\x01" + mth(data[:k]) + mth(data[k:]))


def state_hash(buffers: Iterable[bytes], leaf_bytes: int = LEAF_BYTES) -> bytes:
    """32-byte digest of the state given as a list of byte buffers."""
    return mth(leaves(buffers, leaf_bytes))


def audit_path(m: int, data: Sequence[bytes]) -> List[bytes]:
    """RFC 6962 section 2.1.1 audit path PATH(m, D[n]) for leaf m."""
    n = len(data)
    if n <= 1:
        return []
    k = 1
    while k * 2 < n:
        k *= 2
    if m < k:
        return audit_path(m, data[:k]) + [mth(data[k:])]
    return audit_path(m - k, data[k:]) + [mth(data[:k])]
