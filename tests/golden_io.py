"""Readers for the hand-worked fixtures under tests/golden/ (see each file's
header for the passage it follows)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                yield line


def bits_to_f32(b: int) -> np.float32:
    return np.array([b], dtype=np.uint32).view(np.float32)[0]


def f32_to_bits(x) -> int:
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0])


def quant_cases():
    for line in _lines("quant_rne.txt"):
        xb, sb, q = line.split()
        yield int(xb, 16), int(sb, 16), int(q)


def ftz_cases():
    for line in _lines("ftz_cases.txt"):
        op, a, b, e = line.split()
        yield op, int(a, 16), int(b, 16), int(e, 16)


def canon_cases():
    """Yields (terms float32 array, expected bits)."""
    for line in _lines("canon_discriminators.txt"):
        lhs, rhs = line.split("->")
        toks = lhs.split()
        L = int(toks[0])
        fill = float(toks[1])
        p = np.full(L, fill, dtype=np.float32)
        for t in toks[2:]:
            i, v = t.split(":")
            p[int(i)] = np.float32(float(v))
        yield p, int(rhs.split()[0], 16)


def treefold_cases():
    for line in _lines("treefold_cases.txt"):
        lhs, rhs = line.split("->")
        toks = lhs.split()
        R = int(toks[0])
        vals = np.array([float(v) for v in toks[1:]], dtype=np.float32)
        assert vals.size == R
        yield vals, int(rhs.split()[0], 16)


def sha256_vectors():
    """Yields (message bytes, expected digest bytes)."""
    for line in _lines("sha256_vectors.txt"):
        msg, dig = line.split()
        yield (b"" if msg == "-" else bytes.fromhex(msg)), bytes.fromhex(dig)


def _value(tok: str) -> float:
    """A decimal literal or a signed power of two written as [-]2^e."""
    if "^" in tok:
        neg = tok.startswith("-")
        base, e = tok.lstrip("-").split("^")
        assert base == "2"
        v = 2.0 ** int(e)
        return -v if neg else v
    return float(tok)


def _range(tok: str):
    lo, _, hi = tok.partition("-")
    return int(lo), int(hi) if hi else int(lo)


def attn_order_cases():
    """Yields dicts: name, kind, T, W, Hq, Hkv, row, col, bits, times_c and
    assign = [(tensor, i_lo, i_hi, h, d_lo, d_hi, value)]."""
    for line in _lines("attn_order.txt"):
        toks = line.split()
        name, kind = toks[0], toks[1]
        T, W, Hq, Hkv, row, col = (int(t) for t in toks[2:8])
        exp = toks[8]
        times_c = exp.startswith("c*")
        bits = int(exp[2:] if times_c else exp, 16)
        assign = []
        for a in toks[9:]:
            lhs, val = a.split("=")
            tensor, idx = lhs.split("[")
            i_t, h_t, d_t = idx.rstrip("]").split(",")
            i_lo, i_hi = _range(i_t)
            d_lo, d_hi = _range(d_t)
            assign.append((tensor, i_lo, i_hi, int(h_t), d_lo, d_hi, _value(val)))
        yield dict(name=name, kind=kind, T=T, W=W, Hq=Hq, Hkv=Hkv, row=row, col=col, bits=bits,
                   times_c=times_c, assign=assign)
