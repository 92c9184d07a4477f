"""Host-side helpers around the paged layout: slot arithmetic, KV sizing and
setting up device pools from logical K/V through the library's own
reshape_and_cache.

Pool layout (both K and V): [num_blocks][Hkv][block_size][head_dim].
"""
from __future__ import annotations

import numpy as np
import torch

from . import ops


def slots_for(table_row, positions, block_size):
    """Slots of the given logical positions of one sequence:
    physical block table_row[j // bs] times bs, plus j % bs ("PagedAttention:
    memetakan blok KV logis ke memori fisik tidak kontigu", section "Urutan
    logis dipisahkan dari penempatan fisik")."""
    pos = np.asarray(positions, dtype=np.int64)
    row = np.asarray(table_row, dtype=np.int64)
    return row[pos // block_size] * block_size + pos % block_size


def kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes):
    """Bytes of K and V one token keeps across all layers."""
    return 2 * layers * kv_heads * head_dim * elem_bytes


def alloc_pools(num_blocks, Hkv, block_size, head_dim, dtype, device="cuda", poison=True):
    """K and V pools; poisoned with NaN so that any read of a slot nobody
    wrote shows up in the output."""
    shape = (num_blocks, Hkv, block_size, head_dim)
    if poison:
        k = torch.full(shape, float("nan"), dtype=dtype, device=device)
        v = torch.full(shape, float("nan"), dtype=dtype, device=device)
    else:
        k = torch.empty(shape, dtype=dtype, device=device)
        v = torch.empty(shape, dtype=dtype, device=device)
    return k, v


def all_slots(table, lens, block_size):
    """Slots of every token of every sequence, stacked in logical order."""
    parts = [slots_for(table[s], np.arange(int(L)), block_size) for s, L in enumerate(lens)]
    return np.concatenate(parts) if parts else np.zeros(0, np.int64)


def fill_pools(k_cache, v_cache, k_logical, v_logical, table, lens, block_size, chunk=1 << 20):
    """Write stacked logical K/V [sum L][Hkv][d] into the pools at the slots the
    block table gives, with pa_reshape_and_cache."""
    slots = torch.from_numpy(all_slots(table, lens, block_size)).to(k_cache.device)
    for i in range(0, slots.numel(), chunk):
        sl = slice(i, i + chunk)
        ops.reshape_and_cache(k_logical[sl].to(k_cache.device).contiguous(),
                              v_logical[sl].to(k_cache.device).contiguous(), k_cache, v_cache,
                              slots[sl].contiguous())


def kv_utilization(lens, block_size, reserve_len=None):
    """Fraction of allocated KV slots that hold tokens.

    Paged: every sequence holds ceil(L/bs) blocks, so the unfilled slots are
    less than one block per sequence ("PagedAttention: memetakan blok KV
    logis ke memori fisik tidak kontigu", section "Sisa alokasi dibatasi oleh
    granularitas blok").  Contiguous: every sequence reserves reserve_len
    slots up front, the max-length reservation the pages contrast with paging
    ("Apa itu PagedAttention?", section "Masalah fragmentasi memori KV Cache
    konvensional").  Returns (paged, contiguous or None).
    """
    lens = np.asarray(lens, dtype=np.int64)
    used = int(lens.sum())
    paged = used / float(int(sum(-(-int(L) // block_size) for L in lens)) * block_size)
    contiguous = None
    if reserve_len is not None:
        contiguous = used / float(len(lens) * int(reserve_len))
    return paged, contiguous


def place_prefix_forks(pf, bm_seed, extra_blocks=None):
    """Run the fork step of a shared-prefix batch through the native block
    manager and return where everything lands.

    The system prompt is added once; every user forks it (its prompt blocks
    are shared, refcount B+1) and appends its private history except the
    newest token; the parents each fork a child; then every sequence appends
    one token in ascending id order (users, then children), so a parent whose
    last block is partly filled takes the copy-on-write copy of it and its
    child writes into the shared original ("Apa itu PagedAttention?", section
    "Cara kerja PagedAttention", item 3).

    Returns a dict: num_blocks, table [B+forks][MB] int32, lens [B+forks],
    pairs (copy-on-write (src, dst) list), prompt_slots [P], hist_rows and
    hist_slots (the users' private histories: rows of ``pf.base.k`` and their
    slots), new_slots [B+forks] and the new rows k_new/v_new [B+forks][Hkv][d].
    """
    import torch

    from .block_manager import BlockManager
    w = pf.base
    P, suffix, bs = w.extra["prefix"], w.extra["suffix"], w.bs
    B, nf = w.B, len(pf.parents)
    offs = w.kv_offsets
    need = P // bs + sum(-(-int(x) // bs) for x in suffix)
    NB = int(np.ceil(1.2 * need)) + (2 * nf if extra_blocks is None else extra_blocks)
    bm = BlockManager(NB, bs, seed=bm_seed)
    system = 1 << 40
    prompt_slots = bm.add_seq(system, P)
    hist_slots, hist_rows = [], []
    for s_ in range(B):
        bm.fork(system, s_)
        sl, _ = bm.append_n(s_, int(suffix[s_]) - 1)
        hist_slots.append(sl)
        hist_rows.append(np.arange(offs[s_] + P, offs[s_] + w.lens[s_] - 1))
    children = [(1 << 41) + i for i in range(nf)]
    for par, ch in zip(pf.parents, children):
        bm.fork(int(par), ch)
    order = list(range(B)) + children
    new_slots, pairs = [], []
    for seq in order:
        slot, a, b = bm.append(seq)
        new_slots.append(slot)
        if a >= 0:
            pairs.append((a, b))
    MB = max(len(bm.seq_blocks(s_)) for s_ in order)
    last = torch.from_numpy(offs + w.lens - 1)
    out = dict(num_blocks=NB, table=bm.block_table(order, MB),
               lens=np.array([bm.seq_len(s_) for s_ in order], dtype=np.int64),
               pairs=pairs, prompt_slots=prompt_slots,
               hist_rows=np.concatenate(hist_rows).astype(np.int64),
               hist_slots=np.concatenate(hist_slots).astype(np.int64),
               new_slots=np.asarray(new_slots, dtype=np.int64),
               k_new=torch.cat([w.k[last], pf.k_child]),
               v_new=torch.cat([w.v[last], pf.v_child]), bm=bm)
    return out
