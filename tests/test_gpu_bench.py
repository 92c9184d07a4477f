"""bench.py's GPU arm prints the contract's JSON line: whole-job metric,
roofline of the dominant kernel (live CUDA-event timing, measured peak),
end-to-end value through host buffers, clocks sampled during the timed
region, the kernel launch count and the oracle baseline."""
import importlib.util
import json
import os

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu


def test_default_bench_line(capsys):
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    bench.main(["--steps", "20", "--warmup", "3", "--cpu-sample-seqs", "2"])
    j = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert j["metric"] == bench.METRIC and j["unit"] == "GB/s" and j["n_gpus"] == 1
    assert j["steps"] == 20 and j["warmup"] == 3 and j["value"] > 0 and j["ms_per_step"] > 0
    assert j["config"]["workload"] == bench.WORKLOADS["8b"] and j["dtype"] == "bf16"
    r = j["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert 0 < r["frac"] < 1.5 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    e2e = j["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert j["gpu_launches"] == 3 * 20  # store, decode, merge of split items
    assert "decode_persistent_kernel, tensor-core tile" in j["roofline"]["kernel"]
    assert "sm_mhz" in j["clocks"] and "reasons" in j["clocks"]
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
