"""reshape_and_cache and copy_blocks on the GPU: bit-exact against the
oracle's byte scatter and block copy; copy-on-write through the native block
manager leaves every other branch untouched."""
import numpy as np
import pytest
import torch

import oracle
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


def _host(t):
    """Device tensor -> numpy array of the same bytes (bf16 viewed as int16)."""
    t = t.cpu()
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).numpy()


@pytest.mark.parametrize("dtype,d,bs", [(torch.bfloat16, 128, 16), (torch.float32, 64, 16),
                                        (torch.bfloat16, 64, 32), (torch.bfloat16, 128, 8)])
def test_reshape_and_cache_bit_exact(dtype, d, bs):
    NB, Hkv, T = 40, 4, 150
    g = torch.Generator().manual_seed(1)
    k_new = torch.randn(T, Hkv, d, generator=g).to(dtype)
    v_new = torch.randn(T, Hkv, d, generator=g).to(dtype)
    slots = torch.from_numpy(np.random.default_rng(2).permutation(NB * bs)[:T].astype(np.int64))
    slots[[3, 77]] = -1  # padding entries are skipped
    kc = torch.randn(NB, Hkv, bs, d, generator=g).to(dtype)
    vc = torch.randn(NB, Hkv, bs, d, generator=g).to(dtype)
    k_ref, v_ref = _host(kc).copy(), _host(vc).copy()
    oracle.reshape_and_cache(_host(k_new), _host(v_new), k_ref, v_ref, slots.numpy(), bs)
    kd, vd = kc.to(DEV), vc.to(DEV)
    ops().reshape_and_cache(k_new.to(DEV), v_new.to(DEV), kd, vd, slots.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(_host(kd), k_ref) and np.array_equal(_host(vd), v_ref)


def test_reshape_8b_step_full_pool():
    """The 8B config's per-step store: one new token per sequence (64) into a
    10k-block pool; the whole pool compared byte for byte."""
    w = synth.decode_workload("8b", seed=0)
    from paged_kv_cache_192_gb300.layout import slots_for
    slots = np.array([slots_for(w.table[s], [w.lens[s] - 1], w.bs)[0] for s in range(w.B)])
    g = torch.Generator().manual_seed(4)
    k_new = torch.randn(w.B, w.Hkv, w.d, generator=g).to(w.dtype)
    v_new = torch.randn(w.B, w.Hkv, w.d, generator=g).to(w.dtype)
    kc = torch.zeros(w.num_blocks, w.Hkv, w.bs, w.d, dtype=w.dtype)
    vc = torch.zeros_like(kc)
    k_ref, v_ref = _host(kc).copy(), _host(vc).copy()
    oracle.reshape_and_cache(_host(k_new), _host(v_new), k_ref, v_ref, slots, w.bs)
    kd, vd = kc.to(DEV), vc.to(DEV)
    ops().reshape_and_cache(k_new.to(DEV), v_new.to(DEV), kd, vd,
                            torch.from_numpy(slots).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(_host(kd), k_ref) and np.array_equal(_host(vd), v_ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_copy_blocks_bit_exact(dtype):
    NB, Hkv, bs, d = 30, 8, 16, 128
    g = torch.Generator().manual_seed(5)
    kc = torch.randn(NB, Hkv, bs, d, generator=g).to(dtype)
    vc = torch.randn(NB, Hkv, bs, d, generator=g).to(dtype)
    pairs = np.array([[3, 20], [7, 21], [3, 22], [29, 0]], dtype=np.int64)
    k_ref, v_ref = _host(kc).copy(), _host(vc).copy()
    oracle.copy_blocks(k_ref, v_ref, pairs)
    kd, vd = kc.to(DEV), vc.to(DEV)
    ops().copy_blocks(kd, vd, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(_host(kd), k_ref) and np.array_equal(_host(vd), v_ref)


def test_validate_rejects_duplicate_slots_and_overlapping_pairs():
    from paged_kv_cache_192_gb300._lib import PAError
    kc = torch.zeros(8, 2, 16, 64, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kn = torch.zeros(3, 2, 64, dtype=torch.bfloat16, device=DEV)
    ops().set_validate(True)
    try:
        with pytest.raises(PAError):
            ops().reshape_and_cache(kn, kn, kc, vc, torch.tensor([5, 9, 5], device=DEV))
        with pytest.raises(PAError):
            ops().reshape_and_cache(kn, kn, kc, vc, torch.tensor([5, 9, 8 * 16], device=DEV))
        with pytest.raises(PAError):
            ops().copy_blocks(kc, vc, torch.tensor([[1, 2], [2, 3]], device=DEV))
        ops().reshape_and_cache(kn, kn, kc, vc, torch.tensor([5, -1, 8], device=DEV))
    finally:
        ops().set_validate(False)


def test_fork_cow_leaves_siblings_untouched():
    """Shared-prefix config's fork step: 64 parents each fork a child; parent and
    child append one different token; copy-on-write copies run before the
    stores.  Every other sequence's blocks stay byte-identical, refcounts
    follow the model, and each branch reads back its own new token."""
    from oracle.bm_model import BlockManagerModel
    from paged_kv_cache_192_gb300.block_manager import BlockManager
    cfg = synth.CONFIGS["prefix"]
    Hkv, d, bs, dtype = cfg["Hkv"], cfg["d"], cfg["bs"], cfg["dtype"]
    B, P = 256, cfg["prefix"]
    rng = np.random.default_rng(0)
    suffix = rng.integers(1, 513, size=B)
    NB = int(np.ceil(1.2 * (P // bs + sum(-(-int(x) // bs) for x in suffix)))) + 2 * 64
    bm, model = BlockManager(NB, bs, seed=11), BlockManagerModel(NB, bs, seed=11)
    g = torch.Generator().manual_seed(0)
    kc = torch.randn(NB, Hkv, bs, d, generator=g).to(dtype).to(DEV)
    vc = torch.randn(NB, Hkv, bs, d, generator=g).to(dtype).to(DEV)
    # the system prompt, then 256 users sharing it with private suffixes
    bm.add_seq(1000, P)
    model.add_seq(1000, P)
    for s in range(B):
        bm.fork(1000, s)
        model.fork(1000, s)
        sl, _ = bm.append_n(s, int(suffix[s]))
        assert list(sl) == model.append_n(s, int(suffix[s]))[0]
    assert all(bm.refcount(b) == B + 1 for b in bm.seq_blocks(1000))
    parents = np.sort(rng.choice(B, size=64, replace=False))
    snapshot_k, snapshot_v = kc.clone(), vc.clone()
    pairs, slots, new_k, new_v, writers = [], [], [], [], []
    for i, par in enumerate(parents):
        child = 2000 + i
        bm.fork(int(par), child)
        model.fork(int(par), child)
        for seq in (int(par), child):  # ascending ids: the parent writes first
            slot, a, b = bm.append(seq)
            assert (slot, a, b) == model.append(seq)
            if a >= 0:
                pairs.append((a, b))
            slots.append(slot)
            writers.append(seq)
            new_k.append(torch.randn(Hkv, d, generator=g))
            new_v.append(torch.randn(Hkv, d, generator=g))
    n_cow = sum(1 for par in parents if (P + suffix[par]) % bs != 0)
    assert len(pairs) == n_cow
    if pairs:
        ops().copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int64, device=DEV))
    kn = torch.stack(new_k).to(dtype).to(DEV)
    vn = torch.stack(new_v).to(dtype).to(DEV)
    ops().reshape_and_cache(kn, vn, kc, vc, torch.tensor(slots, dtype=torch.int64, device=DEV))
    torch.cuda.synchronize()
    touched = {b for _, b in pairs} | {s // bs for s in slots}
    untouched = torch.tensor(sorted(set(range(NB)) - touched), device=DEV)
    assert torch.equal(kc[untouched], snapshot_k[untouched])
    assert torch.equal(vc[untouched], snapshot_v[untouched])
    # every copy is a faithful copy of its source apart from the new token
    for (a, b) in pairs:
        slot_in_b = [s for s in slots if s // bs == b]
        mask = torch.ones(bs, dtype=torch.bool)
        for s in slot_in_b:
            mask[s % bs] = False
        assert torch.equal(kc[b][:, mask.to(DEV)], snapshot_k[a][:, mask.to(DEV)])
    # each branch reads back its own token at its own slot
    for i, (seq, slot) in enumerate(zip(writers, slots)):
        blk, off = divmod(slot, bs)
        assert torch.equal(kc[blk, :, off], kn[i])
        assert bm.seq_blocks(seq) == model.blocks[seq]
    for b in range(NB):
        assert bm.refcount(b) == model.ref[b]
