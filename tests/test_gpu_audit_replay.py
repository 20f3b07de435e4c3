"""The audit claim the library exists for, on the GPU: a training step replayed
under a different launch configuration -- other backward kernel, other
reduction segments, other streaming grids, the CUDA-core forward -- gives the
same per-step state hash, and a single flipped input bit gives another.

The step is the three-level replay with the optimiser: per micro-batch scales,
int8 codes, exact forward, canonical-order backward with fused accumulation;
the running sum over shard partials; TreeFold over replicas; clip + AdamW; the
Merkle state hash of (parameters, first moment, second moment)."""
import dataclasses

import numpy as np
import pytest

from bitwise_reproducible_int8_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import bitwise_reproducible_int8_gb300 as R  # noqa: E402
from bitwise_reproducible_int8_gb300 import step as S  # noqa: E402

WL = inputs.Workload("audit_small", 256,
                     (inputs.Linear("a", 192, 128), inputs.Linear("b", 64, 192, silu_input=True)),
                     microbatches=3, replicas=3, w_seed_base=7, x_seed_base=11,
                     description="two linears, 3 micro-batches, 2 shards, 3 replicas, AdamW",
                     shards=2, optimizer=True)

CONFIGS = [
    {},
    {"bwd_kernel": 8, "bwd_segment_log2": 0, "elementwise_blocks": 7, "reduce_block_log2": 2,
     "fwd_path": 0},
    {"bwd_kernel": 1, "bwd_segment_log2": 1, "elementwise_blocks": 1, "reduce_block_log2": 0},
]


def _replay(host, cfg, steps=2, dw_stream=None):
    R.repro_set_launch_cfg(reset=True)
    if cfg:
        R.repro_set_launch_cfg(**cfg)
    try:
        hp = S.HotPathStep(WL, host, dw_stream=dw_stream)
        st = torch.cuda.current_stream()
        hp.prepare(st)
        log = []
        for _ in range(steps):
            hp.run(st)
            torch.cuda.synchronize()
            assert R.repro_device_check() == 0
            log.append(bytes(hp.digest.cpu().numpy()))
        return log
    finally:
        R.repro_set_launch_cfg(reset=True)


def test_replay_under_other_launch_configurations_gives_the_same_hashes():
    host = S.generate_host_inputs(WL)
    logs = [_replay(host, cfg) for cfg in CONFIGS]
    logs.append(_replay(host, {}, dw_stream=True))   # dW on its own stream
    assert logs[0][0] != logs[0][1]            # the state moved
    for other in logs[1:]:
        assert other == logs[0]


def test_one_flipped_input_bit_changes_the_hash():
    host = S.generate_host_inputs(WL)
    base = _replay(host, {}, steps=1)
    dy = [[x.copy() for x in row] for row in host.dY]
    dy[1][2].view(np.uint32)[17, 5] ^= 1       # last micro-batch of the second linear
    tampered = dataclasses.replace(host, dY=dy)
    assert _replay(tampered, {}, steps=1) != base
