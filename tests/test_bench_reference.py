"""The bench's reference arm on CPU: the float64 oracle timed on this host's cores,
printed as one JSON line with the contract's keys; under several ranks only rank 0
prints."""
import argparse
import json

import bench


def _args(steps=1, warmup=0):
    return argparse.Namespace(steps=steps, warmup=warmup, gpus=1, impl="reference")


def test_reference_arm_prints_one_contract_line(capsys):
    bench.run_reference(_args(), rank=0, world=1, budget=2.0)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "queries/s"
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] == 0
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["dtype"] == "f64" and line["vs_baseline"] is None
    assert line["config"]["workload"] == bench.WORKLOAD
    assert 1 <= line["config"]["queries_per_step"] <= 64
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "queries/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing(capsys):
    bench.run_reference(_args(), rank=1, world=2, budget=2.0)
    assert capsys.readouterr().out == ""
