"""Reference model of the paged KV block manager -- TEST INFRASTRUCTURE ONLY.

A deliberately plain Python model, checked step by step against the native
block manager.  It follows the pages:

* KV is kept in fixed-size blocks reached through a per-sequence block table
  that maps logical block i to a physical block anywhere in the pool
  ("PagedAttention: memetakan blok KV logis ke memori fisik tidak kontigu",
  section "Urutan logis dipisahkan dari penempatan fisik").
* A new physical block is taken only when the sequence crosses a block
  boundary, from anywhere in the free pool ("Melihat Lebih Dalam vLLM v0.7",
  section "Blueprint Arsitektur 2", item 3 "Alokasi On-Demand"; "Apa itu
  PagedAttention?", section "Cara kerja PagedAttention", item 2).
* Several sequences may point to one physical block (shared prompt, parallel
  sampling); a block stays shared while its content does not change, and a
  branch that must write into a shared block gets its own copy first
  (copy-on-write) -- "Apa itu PagedAttention?", item 3; nalar.dev, section
  "Sharing blok dapat menghindari duplikasi state KV".
* The waste of a sequence is bounded by one block's granularity (nalar.dev,
  section "Sisa alokasi dibatasi oleh granularitas blok").

Readings where the pages are silent (shared with the native manager because
the two are compared block id by block id):
* free list: a stack; the initial order is 0..NB-1, or a Fisher-Yates shuffle
  driven by SplitMix64 (Steele, Lea, Flood 2014; Vigna's reference constants)
  when a nonzero seed is given; allocation takes the next block of that order;
  freed blocks are pushed back and reused first.
* copy-on-write: the branch that appends into a shared, partly filled last
  block takes the new copy; the last holder writes in place.  A full shared
  last block needs no copy (the new token starts a fresh block).
* failed calls change nothing (out of blocks is checked before any change).
"""
from __future__ import annotations

_M64 = (1 << 64) - 1


class OutOfBlocks(Exception):
    pass


def splitmix64(state: int):
    """SplitMix64 step: returns (new_state, output)."""
    state = (state + 0x9E3779B97F4A7C15) & _M64
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return state, z ^ (z >> 31)


def initial_order(num_blocks: int, seed: int):
    order = list(range(num_blocks))
    if seed:
        st = seed & _M64
        for i in range(num_blocks - 1, 0, -1):
            st, r = splitmix64(st)
            j = r % (i + 1)
            order[i], order[j] = order[j], order[i]
    return order


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int, seed: int = 0):
        self.nb = num_blocks
        self.bs = block_size
        self.free = list(reversed(initial_order(num_blocks, seed)))  # top = end
        self.ref = [0] * num_blocks
        self.blocks: dict[int, list[int]] = {}
        self.length: dict[int, int] = {}

    # -- helpers ---------------------------------------------------------
    def _take(self) -> int:
        b = self.free.pop()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _release(self, b: int):
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            self.free.append(b)

    def _blocks_needed(self, seq: int, n: int) -> int:
        L = self.length[seq]
        bs = self.bs
        need = -(-(L + n) // bs) - (-(-L // bs))
        if n > 0 and L % bs != 0 and self.ref[self.blocks[seq][-1]] > 1:
            need += 1
        return need

    # -- API -------------------------------------------------------------
    def add_seq(self, seq: int, n_tokens: int):
        """New sequence holding n_tokens prompt tokens; returns their slots."""
        if seq in self.blocks or n_tokens < 0:
            raise ValueError("bad sequence")
        nblk = -(-n_tokens // self.bs)
        if nblk > len(self.free):
            raise OutOfBlocks()
        self.blocks[seq] = [self._take() for _ in range(nblk)]
        self.length[seq] = n_tokens
        return [self.slot(seq, j) for j in range(n_tokens)]

    def fork(self, parent: int, child: int):
        if parent not in self.blocks or child in self.blocks:
            raise ValueError("bad sequence")
        self.blocks[child] = list(self.blocks[parent])
        self.length[child] = self.length[parent]
        for b in self.blocks[child]:
            self.ref[b] += 1

    def append(self, seq: int):
        """One new token; returns (slot, cow_src, cow_dst) with -1 for no copy."""
        if seq not in self.blocks:
            raise ValueError("bad sequence")
        if self._blocks_needed(seq, 1) > len(self.free):
            raise OutOfBlocks()
        L = self.length[seq]
        bl = self.blocks[seq]
        src = dst = -1
        if L % self.bs == 0:
            bl.append(self._take())
        elif self.ref[bl[-1]] > 1:
            src = bl[-1]
            dst = self._take()
            self._release(src)
            bl[-1] = dst
        self.length[seq] = L + 1
        return bl[-1] * self.bs + L % self.bs, src, dst

    def append_n(self, seq: int, n: int):
        """n new tokens at once; returns (slots, cow pairs), all or nothing."""
        if seq not in self.blocks or n < 0:
            raise ValueError("bad sequence")
        if self._blocks_needed(seq, n) > len(self.free):
            raise OutOfBlocks()
        slots, pairs = [], []
        for _ in range(n):
            s, a, b = self.append(seq)
            slots.append(s)
            if a >= 0:
                pairs.append((a, b))
        return slots, pairs

    def free_seq(self, seq: int):
        if seq not in self.blocks:
            raise ValueError("bad sequence")
        for b in self.blocks.pop(seq):
            self._release(b)
        del self.length[seq]

    def slot(self, seq: int, j: int) -> int:
        return self.blocks[seq][j // self.bs] * self.bs + j % self.bs

    def block_table(self, seqs, max_blocks: int):
        rows = []
        for s in seqs:
            bl = self.blocks[s]
            if len(bl) > max_blocks:
                raise ValueError("table too narrow")
            rows.append(bl + [0] * (max_blocks - len(bl)))
        return rows

    def num_free(self) -> int:
        return len(self.free)
