"""The reference arm of bench.py runs on the host (the oracle on a bounded
sample), so its JSON line can be checked here without a GPU: one line, every
key of the contract, and the host-only e2e block."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_line_keeps_the_contract():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                          "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True,
                         text=True, timeout=600, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["unit"] == "tokens/s" and d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_oracle_sample_fractions():
    # the CPU baseline times each part of a step on a sample and divides by
    # the sample's share of that part's work: at 2^-0 the sample is the whole
    # step (every fraction 1, nothing extrapolated); at 2^-3 every part's
    # share is about 1/8 (rounded up to whole outputs)
    sys.path.insert(0, ROOT)
    import bench
    from bitwise_reproducible_int8_gb300 import inputs
    from bitwise_reproducible_int8_gb300 import step as S
    wl = inputs.WORKLOADS["tiny"]
    smp = bench.OracleSample(wl, S.generate_host_inputs(wl))
    r0 = smp.run(0)
    assert all(fr == 1.0 for _, fr in r0["parts"].values())
    assert abs(r0["step_s"] - r0["timed_s"]) < 1e-9
    r3 = smp.run(3, threads=1)
    assert r3["threads"] == 1
    for name, (_, fr) in r3["parts"].items():
        if name != "accumulate":       # one micro-batch: nothing to accumulate
            assert 0.125 <= fr < 0.13, (name, fr)
