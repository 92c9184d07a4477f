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
