"""Seeded synthetic inputs shaped like the pages' 1.61B decoder workloads.

This module only draws random numbers; it contains none of the method's
arithmetic (no scale, quantiser, GEMM or reduction).  It is the one module both
the CUDA path's tests/benchmark and the CPU oracle receive their inputs from.

Generation: every tensor is split into fixed blocks of ``BLOCK`` elements; block
``b`` of tensor ``(seed, stream)`` is drawn from a Philox-4x64 generator keyed by
``SeedSequence([seed, stream, b])``.  The bytes therefore do not depend on the
number of host threads used to fill them.

Workload shapes (Open-1B review, onedev.kr/papers/92, sections "How to use" and
"Premises and limits": 16,384-token micro-batches of 4 x 4,096, d_model 2,048,
16 query / 4 KV heads of 128, SwiGLU gate+up fused, FFN width 5,632).  The
pages' pretraining mix is not available; these synthetic tensors stand in for
it.  Distributions: X ~ N(0, 1) (the down projection's input is SiLU(a)*b with
a, b ~ N(0, 1), computed here in fp32), W ~ N(0, 0.02), dY ~ N(0, 1e-3), replica
noise ~ N(0, 1e-5); the second parameter is the standard deviation.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK = 1 << 20

# stream ids (one independent stream per tensor role)
S_X, S_W, S_DY, S_NOISE, S_A, S_B = 1, 2, 3, 4, 5, 6
S_Q, S_K, S_V, S_DO = 7, 8, 9, 10


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def normal(seed: int, stream: int, shape, std: float = 1.0, rows: int | None = None) -> np.ndarray:
    """float32 N(0, std^2) samples, reproducible for (seed, stream, shape).
    With `rows`, only the first `rows` rows are drawn: the same bytes as the
    leading rows of the full tensor."""
    shape = tuple(int(s) for s in shape)
    if rows is not None:
        shape = (min(int(rows), shape[0]),) + shape[1:]
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=np.float32)
    nblk = (n + BLOCK - 1) // BLOCK

    def fill(b: int) -> None:
        lo, hi = b * BLOCK, min(n, (b + 1) * BLOCK)
        rng = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream, b])))
        rng.standard_normal(out=out[lo:hi], dtype=np.float32)
        if std != 1.0:
            np.multiply(out[lo:hi], np.float32(std), out=out[lo:hi])

    if nblk <= 1:
        for b in range(nblk):
            fill(b)
    else:
        with ThreadPoolExecutor(min(_threads(), nblk)) as ex:
            list(ex.map(fill, range(nblk)))
    return out.reshape(shape)


def silu_times_normal(seed: int, shape, rows: int | None = None) -> np.ndarray:
    """SiLU(a) * b with a, b ~ N(0, 1), in fp32 (the down projection's input)."""
    a = normal(seed, S_A, shape, rows=rows)
    b = normal(seed, S_B, shape, rows=rows)
    # SiLU(a) = a / (1 + exp(-a)), evaluated in fp32 on the host
    with np.errstate(over="ignore"):
        s = a / (np.float32(1.0) + np.exp(-a))
    return (s * b).astype(np.float32, copy=False)


# --------------------------------------------------------------------- shapes

@dataclass(frozen=True)
class Linear:
    name: str
    n_out: int      # N: rows of W (output features)
    k_in: int       # K: columns of W (input features)
    silu_input: bool = False


D_MODEL = 2048
FFN = 5632
HEADS_Q, HEADS_KV, HEAD_DIM = 16, 4, 128
TOKENS_PER_MICROBATCH = 4 * 4096

QKV = Linear("qkv", (HEADS_Q + 2 * HEADS_KV) * HEAD_DIM, D_MODEL)      # 3072 x 2048
O_PROJ = Linear("o_proj", D_MODEL, HEADS_Q * HEAD_DIM)                   # 2048 x 2048
GATE_UP = Linear("gate_up", 2 * FFN, D_MODEL)                            # 11264 x 2048
DOWN = Linear("down", D_MODEL, FFN, silu_input=True)                     # 2048 x 5632


@dataclass(frozen=True)
class Workload:
    name: str
    tokens: int                 # M per micro-batch
    linears: tuple
    microbatches: int = 1
    replicas: int = 0           # R for TreeFold (0: no TreeFold)
    w_seed_base: int = 0        # weight i uses seed w_seed_base + i
    x_seed_base: int = 0        # micro-batch j uses seed x_seed_base + j
    description: str = field(default="", compare=False)
    shards: int = 1             # S for the level-2 running sum (1: none)
    optimizer: bool = False     # clip + AdamW on the folded gradient after TreeFold


WORKLOADS = {
    "tiny": Workload("tiny", 64, (Linear("tiny", 128, 256),), 1, 4, 0, 0,
                     "X[64x256], W[128x256], dY[64x128], seed 0; TreeFold over R=4 copies of dW"),
    "attn_out": Workload("attn_out", TOKENS_PER_MICROBATCH, (O_PROJ,), 1, 0, 0, 0,
                         "attention output projection, one 16,384-token micro-batch"),
    "gate_up": Workload("gate_up", TOKENS_PER_MICROBATCH, (GATE_UP,), 1, 0, 0, 0,
                        "fused SwiGLU gate+up projection as one GEMM"),
    "down_accum": Workload("down_accum", TOKENS_PER_MICROBATCH, (DOWN,), 4, 0, 100, 0,
                           "down projection, 4 micro-batches, dW accumulated in order"),
    "block": Workload("block", TOKENS_PER_MICROBATCH, (QKV, O_PROJ, GATE_UP, DOWN), 4, 6, 100, 0,
                      "one GQA decoder block's linears, 4 micro-batches, TreeFold over R=6"),
    # the audit's full three-level replay: micro-batch accumulation, running sum
    # over S = 8 shard partials of this replica (mesh order), TreeFold over R = 6
    "block_audit": Workload("block_audit", TOKENS_PER_MICROBATCH, (QKV, O_PROJ, GATE_UP, DOWN), 4, 6,
                            100, 0, "block linears, 4 micro-batches, 8 shards, 6 replicas, "
                            "then clip + AdamW", 8, True),
    # profiling case: a few GB on the device, TreeFold inputs (6 x 92 MB) larger than L2
    "gate_up_r6": Workload("gate_up_r6", TOKENS_PER_MICROBATCH, (GATE_UP,), 1, 6, 0, 0,
                           "gate+up projection, one micro-batch, TreeFold over R=6"),
    # profiling case for the backward's DRAM traffic: the block's four linears,
    # one micro-batch, no folds -- every backward launch shape of the block
    # step once, about 5 GB on the device
    "block_1mb": Workload("block_1mb", TOKENS_PER_MICROBATCH, (QKV, O_PROJ, GATE_UP, DOWN), 1, 0,
                          100, 0, "block linears, one micro-batch, no TreeFold"),
    # profiling case for the audit calls: the block's four weights (so the hashed
    # state, 541 MB, and the 8 shard partials exceed L2) with one 2,048-token
    # micro-batch, about 3.5 GB on the device
    "audit_profile": Workload("audit_profile", 2048, (QKV, O_PROJ, GATE_UP, DOWN), 1, 6, 100, 0,
                              "block weights, one 2,048-token micro-batch, 8 shards, 6 replicas, "
                              "then clip + AdamW and the state hash", 8, True),
}


def weight(wl: Workload, i: int) -> np.ndarray:
    lin = wl.linears[i]
    return normal(wl.w_seed_base + i, S_W, (lin.n_out, lin.k_in), 0.02)


def activation(wl: Workload, i: int, mb: int, rows: int | None = None) -> np.ndarray:
    lin = wl.linears[i]
    seed = wl.x_seed_base + mb
    if lin.silu_input:
        return silu_times_normal(seed * 16 + i, (wl.tokens, lin.k_in), rows=rows)
    return normal(seed * 16 + i, S_X, (wl.tokens, lin.k_in), 1.0, rows=rows)


def upstream_grad(wl: Workload, i: int, mb: int, rows: int | None = None) -> np.ndarray:
    lin = wl.linears[i]
    seed = wl.x_seed_base + mb
    return normal(seed * 16 + i, S_DY, (wl.tokens, lin.n_out), 1e-3, rows=rows)


def replica_noise(wl: Workload, r: int, n: int) -> np.ndarray:
    return normal(1000 + r, S_NOISE, (n,), 1e-5)


def shard_noise(wl: Workload, s: int, n: int) -> np.ndarray:
    return normal(2000 + s, S_NOISE, (n,), 1e-5)


def small_case(seed: int, M: int, N: int, K: int, x_std=1.0, w_std=0.02, dy_std=1e-3):
    """Random shapes for parity tests: (X[M,K], W[N,K], dY[M,N])."""
    return (normal(seed, S_X, (M, K), x_std), normal(seed, S_W, (N, K), w_std),
            normal(seed, S_DY, (M, N), dy_std))


# ------------------------------------------------------------------ attention

@dataclass(frozen=True)
class AttnWorkload:
    """One micro-batch through an attention layer: `sequences` x `seq_len`
    tokens, grouped-query heads of HEAD_DIM, causal with a sliding window of
    `window` tokens (0: full causal).  q and k stand for the post-QK-norm
    (gainless RMSNorm) vectors, unit RMS per head, so N(0, 1) entries; v ~ N(0, 1);
    the upstream gradient dO ~ N(0, 1e-3)."""
    name: str
    sequences: int
    seq_len: int
    heads_q: int
    heads_kv: int
    window: int
    seed: int
    description: str = field(default="", compare=False)

    @property
    def tokens(self) -> int:
        return self.sequences * self.seq_len


ATTN_WORKLOADS = {
    # the pages' layers: 512-token sliding window, every fifth and the last layer full causal
    "attn_swa": AttnWorkload("attn_swa", 4, 4096, HEADS_Q, HEADS_KV, 512, 300,
                             "one 16,384-token micro-batch (4 x 4096) through a sliding-window "
                             "layer: 16 query / 4 KV heads of 128, window 512"),
    "attn_causal": AttnWorkload("attn_causal", 4, 4096, HEADS_Q, HEADS_KV, 0, 301,
                                "one 16,384-token micro-batch (4 x 4096) through a full-causal "
                                "layer: 16 query / 4 KV heads of 128"),
    "attn_tiny": AttnWorkload("attn_tiny", 1, 130, 4, 2, 64, 302,
                              "130 tokens, 4 query / 2 KV heads, window 64"),
}


def attn_inputs(aw: AttnWorkload):
    """(q [B,T,Hq,128], k [B,T,Hkv,128], v [B,T,Hkv,128], dO [B,T,Hq,128]) float32."""
    B, T = aw.sequences, aw.seq_len
    q = normal(aw.seed, S_Q, (B, T, aw.heads_q, HEAD_DIM))
    k = normal(aw.seed, S_K, (B, T, aw.heads_kv, HEAD_DIM))
    v = normal(aw.seed, S_V, (B, T, aw.heads_kv, HEAD_DIM))
    do = normal(aw.seed, S_DO, (B, T, aw.heads_q, HEAD_DIM), 1e-3)
    return q, k, v, do
