"""pa_swap_blocks: blocks move between the device pool and a pinned host pool
bit-exactly; a sequence swapped out and back in decodes to the same bits."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import device_inputs
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


def test_swap_out_and_in_bit_exact():
    NB, NH, Hkv, bs, d = 40, 24, 8, 16, 128
    g = torch.Generator().manual_seed(3)
    kd = torch.randn(NB, Hkv, bs, d, generator=g).to(torch.bfloat16).to(DEV)
    vd = torch.randn(NB, Hkv, bs, d, generator=g).to(torch.bfloat16).to(DEV)
    kh = torch.zeros(NH, Hkv, bs, d, dtype=torch.bfloat16).pin_memory()
    vh = torch.zeros_like(kh).pin_memory()
    out_pairs = torch.tensor([[3, 0], [17, 5], [39, 23]], dtype=torch.int64, device=DEV)
    ops().swap_blocks(kh, vh, kd, vd, out_pairs)   # device -> host
    torch.cuda.synchronize()
    for s, t in ((3, 0), (17, 5), (39, 23)):
        assert torch.equal(kh[t], kd[s].cpu()) and torch.equal(vh[t], vd[s].cpu())
    back = torch.tensor([[0, 10], [5, 11], [23, 12]], dtype=torch.int64).pin_memory()
    kd2, vd2 = kd.clone(), vd.clone()
    ops().swap_blocks(kd2, vd2, kh, vh, back)      # host -> device, pairs in host memory
    torch.cuda.synchronize()
    # expected: the oracle's byte copies applied to the device pool
    k_ref = kd.cpu().view(torch.int16).numpy().copy()
    v_ref = vd.cpu().view(torch.int16).numpy().copy()
    oracle.copy_blocks(k_ref, v_ref, [[3, 10], [17, 11], [39, 12]])
    assert np.array_equal(kd2.cpu().view(torch.int16).numpy(), k_ref)
    assert np.array_equal(vd2.cpu().view(torch.int16).numpy(), v_ref)


def test_sequence_swap_roundtrip_decodes_identically():
    """Evict one sequence's blocks to host memory, free them, admit it back
    into fresh device blocks (block manager picks them), decode again."""
    from paged_kv_cache_192_gb300.block_manager import BlockManager
    w = synth.decode_workload("8b", seed=31, lens=[300, 77, 1024], num_blocks=200)
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    before = ops().decode(w.q.to(DEV), k_cache, v_cache, table, lens)
    s, L = 0, int(w.lens[0])
    nblk = -(-L // w.bs)
    # host pool managed by its own block manager
    host_bm = BlockManager(64, w.bs, seed=9)
    host_bm.add_seq(100, L)
    host_blocks = host_bm.seq_blocks(100)
    assert len(host_blocks) == nblk
    kh = torch.zeros(64, w.Hkv, w.bs, w.d, dtype=w.dtype).pin_memory()
    vh = torch.zeros_like(kh).pin_memory()
    dev_blocks = w.table[s, :nblk].astype(np.int64)
    ops().swap_blocks(kh, vh, k_cache, v_cache,
                      torch.tensor(np.stack([dev_blocks, host_blocks], 1), device=DEV))
    torch.cuda.synchronize()
    k_cache[torch.from_numpy(dev_blocks).to(DEV)] = float("nan")   # the device copy is gone
    v_cache[torch.from_numpy(dev_blocks).to(DEV)] = float("nan")
    # swap in to the pool's unused blocks
    used = {int(w.table[b, i]) for b in range(w.B) for i in range(-(-int(w.lens[b]) // w.bs))}
    free = [b for b in range(w.num_blocks) if b not in used][:nblk]
    assert len(free) == nblk
    ops().swap_blocks(k_cache, v_cache, kh, vh,
                      torch.tensor(np.stack([host_blocks, free], 1), device=DEV))
    table2 = table.clone()
    table2[s, :nblk] = torch.tensor(free, dtype=torch.int32, device=DEV)
    after = ops().decode(w.q.to(DEV), k_cache, v_cache, table2, lens)
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    assert torch.equal(before, after)


def test_swap_states_through_block_managers():
    """Swap-out / swap-in bookkeeping on both sides: while a sequence is out,
    the host manager holds its blocks and the device manager has released
    them (here another sequence takes and overwrites them); on swap-in the
    device manager hands out blocks again and the sequence decodes to the
    same bits, through the block table the manager builds."""
    from paged_kv_cache_192_gb300.block_manager import BlockManager
    lens = [300, 77, 1024]
    NB, MB = 200, 64
    w = synth.decode_workload("8b", seed=41, lens=lens, num_blocks=NB, max_blocks=MB)
    dev_bm = BlockManager(NB, w.bs, seed=5)
    for i, L in enumerate(lens):
        dev_bm.add_seq(i, L)
    w.table = dev_bm.block_table(np.arange(3), MB)
    k_cache, v_cache, table, lens_d = device_inputs(w, DEV)
    before = ops().decode(w.q.to(DEV), k_cache, v_cache, table, lens_d)
    torch.cuda.synchronize()

    host_bm = BlockManager(80, w.bs, seed=0)
    kh = torch.zeros(80, w.Hkv, w.bs, w.d, dtype=w.dtype).pin_memory()
    vh = torch.zeros_like(kh).pin_memory()
    free0 = dev_bm.num_free()
    # swap out sequence 2 (1024 tokens = 64 blocks)
    dev_blocks = dev_bm.seq_blocks(2)
    host_bm.add_seq(2, lens[2])
    host_blocks = host_bm.seq_blocks(2)
    ops().swap_blocks(kh, vh, k_cache, v_cache,
                      torch.tensor(np.stack([dev_blocks, host_blocks], 1), device=DEV))
    dev_bm.free_seq(2)
    assert dev_bm.num_free() == free0 + len(dev_blocks)
    # meanwhile another sequence takes device blocks and overwrites them
    dev_bm.add_seq(9, 700)
    taken = torch.tensor(dev_bm.seq_blocks(9), device=DEV)
    k_cache[taken] = float("nan")
    v_cache[taken] = float("nan")
    dev_bm.free_seq(9)
    # swap in: fresh device blocks from the manager, host blocks released
    dev_bm.add_seq(2, lens[2])
    new_blocks = dev_bm.seq_blocks(2)
    ops().swap_blocks(k_cache, v_cache, kh, vh,
                      torch.tensor(np.stack([host_blocks, new_blocks], 1), device=DEV))
    host_bm.free_seq(2)
    assert host_bm.num_free() == 80 and dev_bm.num_free() == free0
    table2 = torch.from_numpy(dev_bm.block_table(np.arange(3), MB)).to(DEV)
    after = ops().decode(w.q.to(DEV), k_cache, v_cache, table2, lens_d)
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    assert torch.equal(before, after)
