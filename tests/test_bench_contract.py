"""bench.py's reference arm (the oracle on the host cores) prints the JSON
line the benchmark contract asks for. It needs no GPU, so it runs here on the
tiny workload; the GPU arm's line is checked on the GPU machine by the bench
itself."""
import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_the_contract_line(capsys):
    import bench
    from speculative_decoding_draft_depth_gb300 import synth
    args = argparse.Namespace(steps=2, warmup=1, gpus=1)
    bench.run_reference(synth.config("tiny"), args)
    line = capsys.readouterr().out.strip().splitlines()[-1]
    d = json.loads(line)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "rounds/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # a step is one whole round: the value is the inverse of the step time
    assert abs(d["value"] - 1000.0 / d["ms_per_step"]) <= 1e-3 * d["value"] + 1e-4
    # the same config keys as the GPU arm
    assert d["config"] == bench.config_dict(synth.config("tiny"), 0) | {"l2": d["config"]["l2"]}
    assert set(d["config"]) == {"workload", "l2", "parallelism"}
