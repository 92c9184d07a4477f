"""Native block manager (C++ behind the C ABI) against the Python reference
model, step by step and bit-exact: slots, copy-on-write pairs, block tables,
refcounts and free counts."""
import numpy as np
import pytest

from conftest import read_golden
from oracle.bm_model import BlockManagerModel, OutOfBlocks


@pytest.fixture(scope="module")
def BM():
    from paged_kv_cache_192_gb300 import build
    build.build()
    from paged_kv_cache_192_gb300.block_manager import BlockManager
    return BlockManager


def _same_state(bm, model, seqs):
    assert bm.num_free() == model.num_free()
    for s in seqs:
        assert bm.seq_len(s) == model.length[s]
        assert bm.seq_blocks(s) == model.blocks[s]
    for b in range(model.nb):
        assert bm.refcount(b) == model.ref[b]


@pytest.mark.parametrize("seed", [0, 7, 12345])
def test_random_operations_match_model(BM, seed):
    from paged_kv_cache_192_gb300._lib import OutOfBlocks as NativeOOB
    rng = np.random.default_rng(seed)
    nb, bs = 96, 8
    bm, model = BM(nb, bs, seed=seed), BlockManagerModel(nb, bs, seed=seed)
    live, next_id = [], 0
    for step in range(600):
        op = rng.integers(0, 10)
        try:
            if op <= 1 or not live:
                n = int(rng.integers(0, 40))
                try:
                    ref = model.add_seq(next_id, n)
                except OutOfBlocks:
                    with pytest.raises(NativeOOB):
                        bm.add_seq(next_id, n)
                    continue
                got = bm.add_seq(next_id, n)
                assert list(got) == ref
                live.append(next_id)
                next_id += 1
            elif op == 2:
                parent = live[int(rng.integers(0, len(live)))]
                model.fork(parent, next_id)
                bm.fork(parent, next_id)
                live.append(next_id)
                next_id += 1
            elif op == 3:
                s = live.pop(int(rng.integers(0, len(live))))
                model.free_seq(s)
                bm.free_seq(s)
            elif op <= 6:
                s = live[int(rng.integers(0, len(live)))]
                try:
                    ref = model.append(s)
                except OutOfBlocks:
                    with pytest.raises(NativeOOB):
                        bm.append(s)
                    continue
                assert bm.append(s) == ref
            else:
                s = live[int(rng.integers(0, len(live)))]
                n = int(rng.integers(1, 20))
                try:
                    ref_slots, ref_pairs = model.append_n(s, n)
                except OutOfBlocks:
                    with pytest.raises(NativeOOB):
                        bm.append_n(s, n)
                    continue
                slots, pairs = bm.append_n(s, n)
                assert list(slots) == ref_slots and pairs == ref_pairs
        finally:
            pass
        if step % 50 == 0:
            _same_state(bm, model, live)
    _same_state(bm, model, live)
    if live:
        mb = max(len(model.blocks[s]) for s in live) + 2
        assert bm.block_table(live, mb).tolist() == model.block_table(live, mb)


def test_worked_example_table(BM):
    """Build the nalar.dev worked mapping 0,1,2,3 -> 17,4,29,8 through the
    native manager's slots (blocks are chosen by the free-list order, so pick
    a pool whose order yields those blocks by allocating in sequence)."""
    rows = read_golden("worked_block_table.txt")
    table = [int(x) for k, vals in rows if k == "table_a" for x in vals]
    bs = int(dict(rows)["block_size"][0])
    bm = BM(32, bs)
    # occupy every other block, free them in an order that leaves 17,4,29,8 on top
    bm.add_seq(0, 32 * bs)
    bm.free_seq(0)  # free order pushes 0..31; top of stack is 31
    filler = [b for b in range(32) if b not in table]
    bm2 = BM(32, bs)
    # simulate: take all blocks, then return them so that the requested ones
    # come out first
    for i in range(32):
        bm2.add_seq(100 + i, bs)
    ids = {b: 100 + b for b in range(32)}
    for b in filler:
        bm2.free_seq(ids[b])
    for b in reversed(table):
        bm2.free_seq(ids[b])
    slots = bm2.add_seq(1, 4 * bs)
    assert bm2.seq_blocks(1) == table
    for k, vals in rows:
        if k == "slot_a":
            t, expect = int(vals[0]), int(vals[1])
            assert slots[t] == expect


def test_parallel_sampling_prompt_saving(BM):
    """N=4 sampled outputs share the prompt blocks ('Melihat Lebih Dalam vLLM
    v0.7', 'Berbagi Memori Fisik'): used prompt memory is 1/4 of private copies."""
    bs, P = 16, 512
    bm = BM(2000, bs, seed=3)
    bm.add_seq(0, P)
    for c in (1, 2, 3):
        bm.fork(0, c)
    used = 2000 - bm.num_free()
    assert used == P // bs
    assert 1 - used / (4 * P // bs) == pytest.approx(0.75)


def test_oom_is_reported_and_state_unchanged(BM):
    from paged_kv_cache_192_gb300._lib import OutOfBlocks as NativeOOB
    bm = BM(4, 16)
    bm.add_seq(0, 40)
    free0 = bm.num_free()
    with pytest.raises(NativeOOB):
        bm.append_n(0, 30)
    assert bm.num_free() == free0 and bm.seq_len(0) == 40
    with pytest.raises(NativeOOB):
        bm.add_seq(1, 33)
    assert bm.num_free() == free0


def test_invalid_calls(BM):
    from paged_kv_cache_192_gb300._lib import PAError
    bm = BM(8, 16)
    bm.add_seq(0, 3)
    with pytest.raises(PAError):
        bm.add_seq(0, 3)
    with pytest.raises(PAError):
        bm.fork(5, 6)
    with pytest.raises(PAError):
        bm.append(9)
    with pytest.raises(PAError):
        bm.block_table([0], 0)


def test_copy_on_write_counts_against_the_pool(BM):
    """A diverging branch's copy of a shared, partly filled block is refused
    when the pool is empty, and nothing changes (same rule as the model)."""
    from paged_kv_cache_192_gb300._lib import OutOfBlocks as NativeOOB
    bm = BM(1, 16)
    bm.add_seq(0, 4)
    bm.fork(0, 1)
    state = (bm.num_free(), bm.seq_blocks(0), bm.seq_blocks(1), bm.refcount(0),
             bm.seq_len(0), bm.seq_len(1))
    with pytest.raises(NativeOOB):
        bm.append(0)
    with pytest.raises(NativeOOB):
        bm.append_n(1, 1)
    assert (bm.num_free(), bm.seq_blocks(0), bm.seq_blocks(1), bm.refcount(0),
            bm.seq_len(0), bm.seq_len(1)) == state
    bm.free_seq(1)                      # the last holder then writes in place
    slot, src, dst = bm.append(0)
    assert (src, dst) == (-1, -1) and slot == bm.seq_blocks(0)[0] * 16 + 4


def test_seeded_order_is_the_models(BM):
    """The native free list starts in the model's seeded order (the same
    SplitMix64-driven Fisher-Yates shuffle), block for block."""
    from oracle.bm_model import initial_order
    for seed in (1, 2, 99, 2**40 + 3):
        bm = BM(50, 8, seed=seed)
        bm.add_seq(0, 50 * 8)
        assert bm.seq_blocks(0) == initial_order(50, seed)


def _snapshot(bm, seqs):
    return (bm.num_free(), [(s, bm.seq_len(s), bm.seq_blocks(s)) for s in seqs],
            [bm.refcount(b) for b in range(bm.num_blocks)])


def _apply(m, op):
    kind, *a = op
    if kind == "add":
        return list(m.add_seq(*a))
    if kind == "fork":
        return m.fork(*a)
    if kind == "append":
        return tuple(m.append(*a))
    if kind == "append_n":
        slots, pairs = m.append_n(*a)
        return list(slots), [tuple(p) for p in pairs]
    if kind == "free":
        return m.free_seq(*a)
    raise AssertionError(kind)


def test_host_allocation_failures_leave_state_unchanged(BM):
    """Host fault injection: every call of a script is failed at each of its
    host allocation points in turn.  Each failure raises OutOfBlocks with the
    manager exactly as before (its later allocations still follow the model,
    so the free-list order is untouched too); then the call runs through and
    matches the model."""
    from paged_kv_cache_192_gb300._lib import OutOfBlocks as NativeOOB
    from paged_kv_cache_192_gb300.block_manager import inject_alloc_failure
    script = [("add", 0, 40), ("fork", 0, 1), ("append", 1), ("append_n", 0, 37),
              ("add", 2, 0), ("append", 2), ("fork", 1, 3), ("append", 3), ("free", 0),
              ("append_n", 3, 20), ("add", 4, 9)]
    bm, model = BM(64, 8, seed=4), BlockManagerModel(64, 8, seed=4)
    live = []
    injected = 0
    for op in script:
        k = 0
        while True:
            before = _snapshot(bm, live)
            inject_alloc_failure(k)
            try:
                got = _apply(bm, op)
            except NativeOOB as e:
                assert "host allocation failed" in str(e)
                assert _snapshot(bm, live) == before, (op, k)
                k += 1
                injected += 1
                continue
            finally:
                inject_alloc_failure(-1)
            break
        assert got == _apply(model, op), op
        if op[0] in ("add", "fork"):
            live.append(op[-2] if op[0] == "add" else op[2])
        elif op[0] == "free":
            live.remove(op[1])
        _same_state(bm, model, live)
    assert injected >= len(script)


def test_create_fails_cleanly_under_host_allocation_failure(BM):
    from paged_kv_cache_192_gb300._lib import OutOfBlocks as NativeOOB
    from paged_kv_cache_192_gb300.block_manager import inject_alloc_failure
    for k in range(4):
        inject_alloc_failure(k)
        try:
            with pytest.raises(NativeOOB, match="host allocation failed"):
                BM(32, 16, seed=1)
        finally:
            inject_alloc_failure(-1)
    assert BM(32, 16, seed=1).num_free() == 32
