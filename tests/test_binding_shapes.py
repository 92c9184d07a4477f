"""The Python binding refuses tensors whose shapes do not match the call
before any pointer reaches the library (the kernels size their reads and
writes from these shapes).  CPU only: every check here runs before the
CUDA-tensor check, which is what a well-shaped CPU tensor then meets."""
import pytest
import torch

from paged_kv_cache_192_gb300 import ops

bf16 = torch.bfloat16


def pools(NB=8, Hkv=2, bs=16, d=64):
    return torch.zeros(NB, Hkv, bs, d, dtype=bf16), torch.zeros(NB, Hkv, bs, d, dtype=bf16)


def decode_args(B=3, Hq=4, d=64, MB=4):
    k, v = pools(d=d)
    return dict(q=torch.zeros(B, Hq, d, dtype=bf16), k_cache=k, v_cache=v,
                block_table=torch.zeros(B, MB, dtype=torch.int32),
                context_lens=torch.ones(B, dtype=torch.int32))


@pytest.mark.parametrize("fn", [ops.decode, ops.decode_noalloc])
@pytest.mark.parametrize("bad,msg", [
    (dict(out=torch.zeros(2, 4, 64, dtype=bf16)), "out must have the shape of q"),
    (dict(block_table=torch.zeros(2, 4, dtype=torch.int32)), "block_table must be"),
    (dict(block_table=torch.zeros(12, dtype=torch.int32)), "block_table must be"),
    (dict(context_lens=torch.ones(4, dtype=torch.int32)), "context_lens must be"),
    (dict(q=torch.zeros(3, 4, 128, dtype=bf16)), "head_dim"),
    (dict(v_cache=torch.zeros(8, 2, 8, 64, dtype=bf16)), "same shape"),
    (dict(q=torch.zeros(3, 256, dtype=bf16)), "q must be"),
])
def test_decode_rejects_mismatched_shapes(fn, bad, msg):
    args = decode_args()
    args.update(bad)
    with pytest.raises(ValueError, match=msg):
        fn(**args)


@pytest.mark.parametrize("fn", [ops.decode, ops.decode_noalloc])
def test_decode_shapes_pass_then_device_check(fn):
    with pytest.raises(ValueError, match="CUDA tensor"):
        fn(**decode_args())


@pytest.mark.parametrize("bad,msg", [
    (dict(k_new=torch.zeros(5, 2, 32, dtype=bf16)), "k_new/v_new"),
    (dict(v_new=torch.zeros(4, 2, 64, dtype=bf16)), "k_new/v_new"),
    (dict(slot_mapping=torch.zeros(4, dtype=torch.int64)), "slot_mapping"),
    (dict(v_cache=torch.zeros(4, 2, 16, 64, dtype=bf16)), "same shape"),
])
def test_reshape_and_cache_rejects_mismatched_shapes(bad, msg):
    k, v = pools()
    args = dict(k_new=torch.zeros(5, 2, 64, dtype=bf16), v_new=torch.zeros(5, 2, 64, dtype=bf16),
                k_cache=k, v_cache=v, slot_mapping=torch.zeros(5, dtype=torch.int64))
    args.update(bad)
    with pytest.raises(ValueError, match=msg):
        ops.reshape_and_cache(**args)


@pytest.mark.parametrize("pairs", [torch.zeros(6, dtype=torch.int64),
                                   torch.zeros(3, 3, dtype=torch.int64)])
def test_block_copies_reject_pairs_not_n_by_2(pairs):
    k, v = pools()
    with pytest.raises(ValueError, match=r"pairs must be \[n\]\[2\]"):
        ops.copy_blocks(k, v, pairs)
    k2, v2 = pools(NB=4)
    with pytest.raises(ValueError, match=r"pairs must be \[n\]\[2\]"):
        ops.swap_blocks(k2, v2, k, v, pairs)


def test_swap_rejects_mismatched_pools():
    k, v = pools()
    k2, v2 = pools(NB=4, bs=8)
    with pytest.raises(ValueError, match="like the source pools"):
        ops.swap_blocks(k2, v2, k, v, torch.zeros(1, 2, dtype=torch.int64))


@pytest.mark.parametrize("bad,msg", [
    (dict(query_start=torch.zeros(4, dtype=torch.int32)), "query_start must be"),
    (dict(block_table=torch.zeros(3, 4, dtype=torch.int32)), "block_table must be"),
    (dict(out=torch.zeros(9, 4, 64, dtype=bf16)), "out must have the shape of q"),
    (dict(q=torch.zeros(10, 4, 128, dtype=bf16)), "head_dim"),
])
def test_prefill_rejects_mismatched_shapes(bad, msg):
    k, v = pools()
    args = dict(q=torch.zeros(10, 4, 64, dtype=bf16), k_cache=k, v_cache=v,
                block_table=torch.zeros(2, 4, dtype=torch.int32),
                query_start=torch.tensor([0, 4, 10], dtype=torch.int32),
                context_lens=torch.tensor([20, 30], dtype=torch.int32), max_query_len=6)
    args.update(bad)
    with pytest.raises(ValueError, match=msg):
        ops.prefill_chunk(**args)
