"""Pins of the reference block-manager model (oracle/bm_model.py) against
what the pages state, independent of the native block manager."""
import numpy as np
import pytest

from oracle.bm_model import BlockManagerModel, OutOfBlocks, initial_order, splitmix64


def test_splitmix64_reference_values():
    """SplitMix64 from seed 0: first outputs as published with the algorithm
    (Vigna's splitmix64.c test values)."""
    st, a = splitmix64(0)
    st, b = splitmix64(st)
    st, c = splitmix64(st)
    assert (a, b, c) == (0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F)


def test_initial_order_is_a_permutation():
    o = initial_order(1000, 42)
    assert sorted(o) == list(range(1000)) and o != list(range(1000))
    assert initial_order(10, 0) == list(range(10))


def test_waste_bounded_by_block_granularity():
    """nalar.dev, 'Sisa alokasi dibatasi oleh granularitas blok': the unfilled
    capacity of a sequence is less than one block."""
    rng = np.random.default_rng(0)
    bm = BlockManagerModel(4096, 16, seed=5)
    for s in range(40):
        bm.add_seq(s, int(rng.integers(0, 100)))
    for _ in range(2000):
        s = int(rng.integers(0, 40))
        bm.append(s)
    for s in range(40):
        slack = len(bm.blocks[s]) * bm.bs - bm.length[s]
        assert 0 <= slack < bm.bs


def test_parallel_sampling_stores_prompt_once():
    """'Melihat Lebih Dalam vLLM v0.7', 'Berbagi Memori Fisik': N=4 outputs of
    one prompt point at the same prompt blocks, saving up to 75% of prompt
    memory."""
    bs, P = 16, 256
    bm = BlockManagerModel(1000, bs)
    bm.add_seq(0, P)
    for c in (1, 2, 3):
        bm.fork(0, c)
    used = 1000 - bm.num_free()
    private = 4 * P // bs
    assert used == P // bs
    assert 1 - used / private == pytest.approx(0.75)
    assert all(bm.ref[b] == 4 for b in bm.blocks[0])


def test_copy_on_write_first_writer_copies():
    bs = 16
    bm = BlockManagerModel(64, bs)
    bm.add_seq(0, 20)            # blocks: full + 4 tokens in the last
    bm.fork(0, 1)
    shared_last = bm.blocks[0][-1]
    slot, src, dst = bm.append(0)  # first writer into the shared partial block
    assert src == shared_last and dst != shared_last
    assert bm.blocks[0][-1] == dst and bm.blocks[1][-1] == shared_last
    assert bm.ref[shared_last] == 1 and bm.ref[dst] == 1
    assert slot == dst * bs + 20 % bs
    slot, src, dst = bm.append(1)  # last holder writes in place
    assert (src, dst) == (-1, -1) and slot == shared_last * bs + 4
    assert bm.ref[bm.blocks[0][0]] == 2  # the full first block stays shared


def test_full_shared_block_needs_no_copy():
    bm = BlockManagerModel(64, 16)
    bm.add_seq(0, 32)
    bm.fork(0, 1)
    _, src, dst = bm.append(1)
    assert (src, dst) == (-1, -1)
    assert bm.ref[bm.blocks[1][0]] == 2 and bm.ref[bm.blocks[1][2]] == 1


def test_out_of_blocks_leaves_state_unchanged():
    bm = BlockManagerModel(4, 16)
    bm.add_seq(0, 40)  # 3 blocks
    before = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.blocks.items()})
    with pytest.raises(OutOfBlocks):
        bm.append_n(0, 30)  # needs 2 more blocks, 1 free
    with pytest.raises(OutOfBlocks):
        bm.add_seq(1, 17)
    assert (bm.free, bm.ref, bm.blocks) == before


def test_freed_blocks_are_reused_first():
    bm = BlockManagerModel(8, 4)
    bm.add_seq(0, 8)
    blocks = list(bm.blocks[0])
    bm.free_seq(0)
    bm.add_seq(1, 4)
    assert bm.blocks[1] == [blocks[-1]]


def test_copy_on_write_counts_against_the_pool():
    """The copy a diverging branch needs is a new block like any other: with
    the pool exhausted the append is refused and nothing changes."""
    bm = BlockManagerModel(1, 16)
    bm.add_seq(0, 4)   # the only block, partly filled
    bm.fork(0, 1)
    before = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.blocks.items()},
              dict(bm.length))
    with pytest.raises(OutOfBlocks):
        bm.append(0)
    with pytest.raises(OutOfBlocks):
        bm.append_n(1, 1)
    assert (bm.free, bm.ref, bm.blocks, bm.length) == before


def test_shuffled_order_reaches_every_permutation():
    """Fisher-Yates (swap with j uniform in [0, i]) can produce every
    permutation: over many seeds all 3! orders of three blocks appear, each
    about equally often.  (Drawing j from [0, i) instead, Sattolo's variant,
    gives only the two cyclic orders.)"""
    counts = {}
    for seed in range(1, 1201):
        o = tuple(initial_order(3, seed))
        counts[o] = counts.get(o, 0) + 1
    assert len(counts) == 6
    assert all(150 <= c <= 250 for c in counts.values()), counts
