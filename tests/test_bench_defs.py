"""The measurement definitions bench.py reports against: algorithmic decode
bytes, causal prefill flops, and the comment-insensitive source key of the
counter records (CPU only)."""
import importlib.util
import os

import numpy as np
import pytest
import torch

from conftest import ROOT


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_decode_bytes_by_hand(bench):
    # 2 sequences of 5 and 17 tokens, 4 query / 2 KV heads, d 64, bf16, 16-token blocks
    kv = (5 + 17) * 2 * 2 * 64 * 2          # K and V rows, once per KV head
    q_out = 2 * 2 * 4 * 64 * 2              # q and out of 2 sequences
    tables = (1 + 2) * 4                    # block-table entries read
    lens = 2 * 4                            # context lengths
    assert bench.decode_bytes([5, 17], 2, 4, 2, 64, 16, torch.bfloat16) == kv + q_out + tables + lens


def test_decode_bytes_of_the_8b_batch(bench):
    from paged_kv_cache_192_gb300 import synth
    w = synth.decode_workload("8b", seed=0)
    assert bench.decode_bytes(w.lens, w.B, w.Hq, w.Hkv, w.d, w.bs, w.dtype) == 564_951_004


def test_prefill_flops_brute_force(bench):
    rng = np.random.default_rng(3)
    Hq, d = 4, 16
    for _ in range(5):
        priors = [int(x) for x in rng.integers(0, 40, size=3)]
        n_new = [int(x) for x in rng.integers(1, 20, size=3)]
        pairs = sum(1 for P, n in zip(priors, n_new) for i in range(n) for j in range(P + i + 1))
        # per (query, key, head): 2 d flops for q.k and 2 d for p*v
        assert bench.prefill_flops(priors, n_new, Hq, d) == pairs * Hq * 4 * d


def test_prefill_flops_of_the_mixed_batch(bench):
    from paged_kv_cache_192_gb300 import synth
    _, pre = synth.mixed_workload(seed=0)
    flops = bench.prefill_flops(pre.extra["prior"], [pre.extra["chunk"]] * len(pre.lens), pre.Hq, pre.d)
    assert flops == 74_675_388_416


def test_source_key_ignores_comments_only(bench, tmp_path, monkeypatch):
    csrc = tmp_path / "paged_kv_cache_192_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "a.cu").write_text("int f() { return 1; }  // one\n/* block\n comment */\n")
    k1 = bench.source_sha1("a.cu")
    (csrc / "a.cu").write_text("int f() { return 1; }  // changed\n/* other */\n")
    assert bench.source_sha1("a.cu") == k1
    (csrc / "a.cu").write_text("int f() { return 2; }\n")
    assert bench.source_sha1("a.cu") != k1


def test_reference_arm_prints_the_contract_line(bench, capsys):
    """bench.py --impl reference: the fp64 oracle on the host cores, one JSON
    line with the same metric and the keys the contract names."""
    import json
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-sample-seqs", "2"])
    line = capsys.readouterr().out.strip().splitlines()[-1]
    j = json.loads(line)
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC and j["unit"] == "GB/s"
    assert j["value"] > 0 and j["higher_is_better"] is True and j["vs_baseline"] is None
    for k in ("n_gpus", "steps", "warmup", "ms_per_step", "scaling", "dtype", "data", "config"):
        assert k in j
    assert j["config"]["workload"] == bench.WORKLOADS["8b"]
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == j["value"] and cb["sample"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["h2d_bytes_per_step"] == 0
    assert e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_follows_the_workload(bench, capsys):
    """--impl reference --workload prefix times the oracle on that workload's
    sequences (256 sharing a 1024-token prompt), not on the default batch."""
    import json
    bench.main(["--impl", "reference", "--workload", "prefix", "--steps", "1", "--warmup", "3",
                "--cpu-sample-seqs", "2"])
    j = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert j["config"]["workload"] == bench.WORKLOADS["prefix"]
    assert j["config"]["B"] == 256 and j["value"] > 0


def test_unique_kv_bytes_counts_shared_blocks_once(bench):
    """Two sequences sharing a 2-block prompt (blocks 7, 3) plus private
    blocks: 5 distinct blocks are read; padding entries past a sequence's
    length do not count."""
    table = np.array([[7, 3, 9, 0], [7, 3, 4, 11]], dtype=np.int32)
    lens = [40, 56]          # 16-token blocks: 3 and 4 blocks
    per_block = 2 * 16 * 64 * 2 * 2   # Hkv * bs * d * es * (K and V)
    assert bench.unique_kv_bytes(table, lens, 16, 2, 64, 2) == 5 * per_block
    assert bench.unique_kv_bytes(table, [1, 1], 16, 2, 64, 2) == 1 * per_block

