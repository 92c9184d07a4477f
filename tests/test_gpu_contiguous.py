"""pa_decode_contiguous (the paging-overhead control: the same decode over a
plain contiguous [B][Hkv][max_len][d] cache, no block table) against the
fp64 oracle; unwritten slots of the reservation are NaN so a read of one
shows in the output."""
import numpy as np
import pytest
import torch

from gpu_util import compare, device_inputs, oracle_decode_all
from paged_kv_cache_192_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_192_gb300 import build
    build.build()


def ops():
    from paged_kv_cache_192_gb300 import ops as o
    return o


def contiguous_inputs(w, max_len):
    """K/V reservations [B][Hkv][max_len][d]: each sequence's logical rows,
    NaN past its length."""
    k = torch.full((w.B, w.Hkv, max_len, w.d), float("nan"), dtype=w.dtype)
    v = torch.full_like(k, float("nan"))
    offs = w.kv_offsets
    for b in range(w.B):
        L = int(w.lens[b])
        k[b, :, :L] = w.k[offs[b]:offs[b] + L].transpose(0, 1)
        v[b, :, :L] = w.v[offs[b]:offs[b] + L].transpose(0, 1)
    return k.to(DEV), v.to(DEV)


def run(w, max_len, partition_tokens=0):
    k, v = contiguous_inputs(w, max_len)
    lens = torch.from_numpy(w.lens.astype(np.int32)).to(DEV)
    out = ops().decode_contiguous(w.q.to(DEV), k, v, lens, partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    return out


def test_8b_shape_contiguous_full_size():
    """The 8B-shaped batch (64 sequences, L ~ U[128,4096], 32/8 heads) in
    4096-token reservations: every output against the oracle and within the
    error bound of the paged decode of the same batch."""
    w = synth.decode_workload("8b", seed=0)
    out = run(w, 4096)
    ref = oracle_decode_all(w)
    compare(out.double().cpu().numpy(), ref, torch.bfloat16, "contiguous 8b")
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    paged = ops().decode(w.q.to(DEV), k_cache, v_cache, table, lens)
    torch.cuda.synchronize()
    compare(paged.double().cpu().numpy(), ref, torch.bfloat16, "paged 8b")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (8, 2), (16, 2)])
def test_contiguous_ragged(dtype, d, Hq, Hkv):
    """Ragged lengths around tile and partition edges (45 sequences, 64-token
    partitions so long ones split) in 320-token reservations, both tiles."""
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 300] * 3
    w = synth.decode_workload("8b", seed=4, lens=lens, Hq=Hq, Hkv=Hkv, d=d, dtype=dtype)
    out = run(w, 320, partition_tokens=64)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), dtype, f"contig d{d} {Hq}/{Hkv}")


def test_contiguous_long_groups_of_8():
    """Long contexts (4 sequences up to 32k tokens, 64 query / 8 KV heads) in
    32768-token reservations: items split over many warps."""
    w = synth.decode_workload("70b", seed=2, B=4)
    out = run(w, 32768, partition_tokens=512)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, "contig 70b")


def test_contiguous_rejects_bad_reservation():
    from paged_kv_cache_192_gb300._lib import PAError
    w = synth.decode_workload("8b", seed=1, lens=[40, 20])
    k = torch.zeros(2, 8, 48, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(PAError):
        ops().decode_contiguous(w.q.to(DEV), k, k.clone(),
                                torch.tensor([40, 20], dtype=torch.int32, device=DEV))
