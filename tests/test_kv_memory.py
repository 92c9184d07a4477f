"""KV-cache memory arithmetic against the figures the pages print, and the
waste of a contiguous max-length reservation against paged allocation."""
import pytest

from conftest import read_golden


def _golden():
    return {k: float(v[0]) for k, v in read_golden("kv_memory_70b.txt")}


def test_70b_sequence_is_about_1_3_gb():
    g = _golden()
    from paged_kv_cache_192_gb300.layout import kv_bytes_per_token
    per_tok = kv_bytes_per_token(int(g["layers"]), int(g["kv_heads"]), int(g["head_dim"]),
                                 int(g["elem_bytes"]))
    assert per_tok == 327680  # 2 x 80 x 8 x 128 x 2 bytes
    seq_gb = per_tok * g["tokens"] / 1e9
    assert seq_gb == pytest.approx(g["page_gb_per_seq"], rel=g["rel_tol"])
    users_gb = seq_gb * g["users"]
    assert users_gb == pytest.approx(g["page_gb_users"], rel=g["rel_tol"])


def test_300_of_4096_reservation_waste():
    """'KV Cache and PagedAttention: Why Your LLM Server Slows Down', 'Traditional
    memory management fails': 300 used of 4096 reserved wastes 93%; 16-token
    blocks waste less than one block."""
    used, reserved, bs = 300, 4096, 16
    assert round(100 * (reserved - used) / reserved) == 93
    paged = -(-used // bs) * bs
    assert 0 <= paged - used < bs


def test_kv_utilization_closed_forms():
    from paged_kv_cache_192_gb300.layout import kv_utilization
    # one 300-token sequence, 16-token blocks, 4096 reserved (the pages' example)
    paged, contig = kv_utilization([300], 16, 4096)
    assert paged == pytest.approx(300 / 304) and contig == pytest.approx(300 / 4096)
    # full blocks waste nothing; the waste is always < one block per sequence
    assert kv_utilization([32, 64], 16)[0] == 1.0
    lens = [1, 17, 31, 100]
    paged, _ = kv_utilization(lens, 16)
    assert sum(lens) / paged - sum(lens) < 16 * len(lens)


def test_kv_utilization_8b_config():
    """8B-shaped batch (L ~ U[128,4096]): paged keeps ~99.6% of the slots
    busy, a 4096-token reservation ~52%."""
    from paged_kv_cache_192_gb300 import synth
    from paged_kv_cache_192_gb300.layout import kv_utilization
    w = synth.decode_workload("8b", seed=0)
    paged, contig = kv_utilization(w.lens, 16, 4096)
    assert 0.99 < paged < 1.0
    assert 0.45 < contig < 0.6
