"""Beam-search style use of the block manager: multi-way forks (refcounts
above 2), branches dying and their blocks recycled, copy-on-write as beams
diverge ("Apa itu PagedAttention?", section "Cara kerja PagedAttention", item
3: parallel sampling / beam search share blocks; "Melihat Lebih Dalam vLLM
v0.7", section "Berbagi Memori Fisik").  Native manager against the Python
model, step by step, plus invariants that hold at every step."""
import numpy as np
import pytest

from oracle.bm_model import BlockManagerModel


@pytest.fixture(scope="module")
def BM():
    from paged_kv_cache_192_gb300 import build
    build.build()
    from paged_kv_cache_192_gb300.block_manager import BlockManager
    return BlockManager


def _invariants(model):
    # refcount of a block == number of live sequences whose table holds it
    count = [0] * model.nb
    for bl in model.blocks.values():
        for b in bl:
            count[b] += 1
    assert count == model.ref
    # free list holds exactly the unreferenced blocks, once each
    assert sorted(model.free) == [b for b in range(model.nb) if model.ref[b] == 0]


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_beam_search_fork_and_prune(BM, seed):
    rng = np.random.default_rng(seed)
    nb, bs, width = 512, 16, 4
    bm, model = BM(nb, bs, seed=seed), BlockManagerModel(nb, bs, seed=seed)
    prompt = int(rng.integers(20, 200))
    assert list(bm.add_seq(0, prompt)) == model.add_seq(0, prompt)
    beams, next_id = [0], 1
    for c in range(1, width):          # 4 beams share the prompt (refcount 4)
        bm.fork(0, c)
        model.fork(0, c)
        beams.append(c)
    next_id = width
    assert max(model.ref) == width
    for step in range(60):
        for b in sorted(beams):         # every beam appends one token (CoW if shared)
            assert bm.append(b) == model.append(b)
        # prune half the beams, refill by forking survivors
        rng.shuffle(beams)
        dead, live = beams[: width // 2], beams[width // 2:]
        for d in dead:
            bm.free_seq(d)
            model.free_seq(d)
        new = []
        for s in live:
            bm.fork(s, next_id)
            model.fork(s, next_id)
            new.append(next_id)
            next_id += 1
        beams = live + new
        _invariants(model)
        assert bm.num_free() == model.num_free()
        for s in beams:
            assert bm.seq_blocks(s) == model.blocks[s]
    for s in beams:
        bm.free_seq(s)
        model.free_seq(s)
    assert bm.num_free() == model.num_free() == nb  # nothing leaks


def test_shared_prefix_memory_saving_grows_with_beams(BM):
    """Stored prompt blocks stay constant while beams multiply."""
    bs, P = 16, 320
    for n in (1, 2, 4, 8):
        bm = BM(1000, bs)
        bm.add_seq(0, P)
        for c in range(1, n):
            bm.fork(0, c)
        assert 1000 - bm.num_free() == P // bs
