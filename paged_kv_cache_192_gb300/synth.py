"""Seeded synthetic workloads for tests and benchmarks.

This module only draws inputs: context lengths, query/key/value values and
the physical placement of each sequence's logical blocks in the pool.  It
holds none of the method's arithmetic (no attention, no slot rule, no cache
layout): both the CUDA path and the fp64 oracle receive what it draws.

Recipe (every config; seed defaults to 0):
* lengths: numpy PCG64(seed), uniform integers in the config's range
  (inclusive), or the fixed list of the tiny config;
* values: torch generator seeded with seed+1, i.i.d. N(0,1), rounded to the
  config's dtype once (bf16 round-to-nearest-even, or fp32); the CPU
  generator by default (tests), the CUDA one where a benchmark only needs a
  multi-GB batch quickly (it then draws a different, equally seeded stream);
* placement: numpy PCG64(seed+2) permutation of the pool's block ids, handed
  out to sequences in order; the pool is 1.2x the blocks needed unless the
  config fixes it (tiny: 32 blocks).  Blocks no sequence owns stay unused.

The K/V histories are LOGICAL: ``k[kv_offsets[s] + j]`` is token j of
sequence s, shape [sum L][Hkv][d].  The shapes mirror Llama-3-8B/70B GQA
attention layers (head counts and head dim only; no weights).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

CONFIGS = {
    # 4 sequences, fp32, MHA, head_dim 64, 16-token blocks in a 32-block pool
    "tiny": dict(lens=[5, 17, 33, 64], Hq=4, Hkv=4, d=64, bs=16, num_blocks=32,
                 dtype=torch.float32),
    # Llama-3-8B-shaped GQA decode
    "8b": dict(B=64, len_range=(128, 4096), Hq=32, Hkv=8, d=128, bs=16, dtype=torch.bfloat16),
    # shared system prompt of 1024 tokens + private suffixes, then 64 forks
    "prefix": dict(B=256, prefix=1024, suffix_range=(1, 512), forks=64, Hq=32, Hkv=8, d=128,
                   bs=16, dtype=torch.bfloat16),
    # Llama-3-70B-shaped long-context decode, split into 512-token partitions
    "70b": dict(B=32, len_range=(16384, 32768), Hq=64, Hkv=8, d=128, bs=32,
                partition=512, dtype=torch.bfloat16),
    # continuous batch: 128 decodes + 4 chunked-prefill requests of 512 tokens
    "mixed": dict(B=128, len_range=(256, 8192), R=4, chunk=512, prior_range=(0, 3584),
                  Hq=32, Hkv=8, d=128, bs=16, dtype=torch.bfloat16),
}


@dataclass
class Workload:
    """Logical inputs of one batch plus the physical placement of its blocks."""

    name: str
    Hq: int
    Hkv: int
    d: int
    bs: int
    dtype: torch.dtype
    lens: np.ndarray            # [B] context length of each sequence (new tokens included)
    q_counts: np.ndarray        # [B] query rows per sequence (1 for decode)
    q: torch.Tensor             # [sum q_counts][Hq][d]
    k: torch.Tensor             # [sum lens][Hkv][d] logical K histories, stacked
    v: torch.Tensor             # [sum lens][Hkv][d]
    table: np.ndarray           # [B][max_blocks] int32, physical block of each logical block
    num_blocks: int
    extra: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return len(self.lens)

    @property
    def kv_offsets(self) -> np.ndarray:
        off = np.zeros(self.B, dtype=np.int64)
        off[1:] = np.cumsum(self.lens)[:-1]
        return off

    @property
    def max_blocks(self) -> int:
        return self.table.shape[1]


def _values(shape, dtype, gen, device="cpu"):
    """N(0,1) values drawn by `gen` on the generator's own device, rounded to
    dtype once, then moved to `device`."""
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=gen.device)
    return x.to(dtype).to(device)


def _generator(seed, gen_device):
    return torch.Generator(device=gen_device).manual_seed(seed)


def _blocks_of(lens, bs):
    return [(int(L) + bs - 1) // bs for L in lens]


def place(blocks_per_seq, num_blocks, rng, max_blocks=None):
    """Random physical placement: a permutation of the pool handed out in order."""
    total = sum(blocks_per_seq)
    assert total <= num_blocks
    perm = rng.permutation(num_blocks)
    mb = max_blocks or max(max(blocks_per_seq), 1)
    table = np.zeros((len(blocks_per_seq), mb), dtype=np.int32)
    pos = 0
    for s, n in enumerate(blocks_per_seq):
        table[s, :n] = perm[pos:pos + n]
        pos += n
    return table


def pool_size(blocks_per_seq, factor=1.2):
    return int(np.ceil(factor * sum(blocks_per_seq)))


def decode_workload(name="8b", seed=0, B=None, lens=None, Hq=None, Hkv=None, d=None, bs=None,
                    dtype=None, num_blocks=None, max_blocks=None, device="cpu", gen_device="cpu"):
    """Decode batch of config ``name`` (one query per sequence), with overrides.

    gen_device="cuda" draws the values with the CUDA generator (same recipe,
    different stream of numbers) -- used to set up multi-GB batches quickly."""
    cfg = dict(CONFIGS[name])
    Hq = Hq or cfg["Hq"]
    Hkv = Hkv or cfg["Hkv"]
    d = d or cfg["d"]
    bs = bs or cfg["bs"]
    dtype = dtype or cfg["dtype"]
    rng_len = np.random.Generator(np.random.PCG64(seed))
    if lens is None:
        if "lens" in cfg:
            lens = cfg["lens"]
        else:
            lo, hi = cfg["len_range"]
            lens = rng_len.integers(lo, hi + 1, size=B or cfg["B"])
    lens = np.asarray(lens, dtype=np.int64)
    nblk = _blocks_of(lens, bs)
    if num_blocks is None:
        num_blocks = cfg.get("num_blocks") if "lens" in cfg and B is None else None
        num_blocks = num_blocks or pool_size(nblk)
    if max_blocks is None:
        max_blocks = max(nblk) if "len_range" not in cfg else (cfg["len_range"][1] + bs - 1) // bs
        max_blocks = max(max_blocks, max(nblk))
    table = place(nblk, num_blocks, np.random.Generator(np.random.PCG64(seed + 2)), max_blocks)
    gen = _generator(seed + 1, gen_device)
    n_kv = int(lens.sum())
    q = _values((len(lens), Hq, d), dtype, gen, device)
    k = _values((n_kv, Hkv, d), dtype, gen, device)
    v = _values((n_kv, Hkv, d), dtype, gen, device)
    return Workload(name, Hq, Hkv, d, bs, dtype, lens, np.ones(len(lens), np.int64), q, k, v,
                    table, num_blocks)


def prefix_workload(seed=0, B=None, prefix=None, suffix_range=None, device="cpu"):
    """Shared-prefix decode batch.

    Every sequence starts with the same ``prefix`` tokens (one system prompt)
    followed by a private suffix.  ``table`` points all sequences at the same
    physical prefix blocks; ``extra['private_table']`` places a private copy
    of the prefix for every sequence in a second, larger pool
    (``extra['private_num_blocks']`` blocks) for the sharing-equivalence check.
    """
    cfg = CONFIGS["prefix"]
    B = B or cfg["B"]
    P = cfg["prefix"] if prefix is None else prefix
    lo, hi = suffix_range or cfg["suffix_range"]
    Hq, Hkv, d, bs, dtype = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["bs"], cfg["dtype"]
    rng_len = np.random.Generator(np.random.PCG64(seed))
    suffix = rng_len.integers(lo, hi + 1, size=B).astype(np.int64)
    lens = P + suffix
    gen = torch.Generator().manual_seed(seed + 1)
    q = _values((B, Hq, d), dtype, gen, device)
    kp = _values((P, Hkv, d), dtype, gen, device)
    vp = _values((P, Hkv, d), dtype, gen, device)
    ks = _values((int(suffix.sum()), Hkv, d), dtype, gen, device)
    vs = _values((int(suffix.sum()), Hkv, d), dtype, gen, device)
    # logical histories: prefix then the sequence's own suffix
    k_parts, v_parts, pos = [], [], 0
    for s in range(B):
        n = int(suffix[s])
        k_parts += [kp, ks[pos:pos + n]]
        v_parts += [vp, vs[pos:pos + n]]
        pos += n
    k = torch.cat(k_parts)
    v = torch.cat(v_parts)
    # shared placement: prefix blocks once, suffix blocks private
    n_pre = (P + bs - 1) // bs
    assert P % bs == 0, "the shared prefix must fill whole blocks"
    n_suf = [(int(x) + bs - 1) // bs for x in suffix]
    mb = n_pre + (hi + bs - 1) // bs + 1
    nb_shared = pool_size([n_pre] + n_suf)
    perm = np.random.Generator(np.random.PCG64(seed + 2)).permutation(nb_shared)
    table = np.zeros((B, mb), dtype=np.int32)
    table[:, :n_pre] = perm[:n_pre]
    pos = n_pre
    for s in range(B):
        table[s, n_pre:n_pre + n_suf[s]] = perm[pos:pos + n_suf[s]]
        pos += n_suf[s]
    nb_private = pool_size([n_pre + x for x in n_suf])
    private = place([n_pre + x for x in n_suf], nb_private,
                    np.random.Generator(np.random.PCG64(seed + 3)), mb)
    w = Workload("prefix", Hq, Hkv, d, bs, dtype, lens, np.ones(B, np.int64), q, k, v, table,
                 nb_shared)
    w.extra.update(prefix=P, suffix=suffix, private_table=private,
                   private_num_blocks=nb_private, prefix_blocks=n_pre)
    return w


@dataclass
class PrefixForks:
    """The shared-prefix batch at its fork step (parallel sampling).

    ``base`` is the pre-fork batch of prefix_workload: B users sharing one
    system prompt, each with a private suffix whose last token is the newest
    one.  ``parents`` (seeded, sorted) each fork one child; every child then
    appends its own new token (``k_child``/``v_child``, query ``q_child``)
    while its parent appends the parent's newest token.  Child i's logical
    history is therefore its parent's history without the newest token,
    followed by the child's own token.
    """

    base: Workload
    parents: np.ndarray          # [forks] user index of each child's parent
    k_child: torch.Tensor        # [forks][Hkv][d]
    v_child: torch.Tensor
    q_child: torch.Tensor        # [forks][Hq][d]

    def logical(self) -> Workload:
        """All B + forks sequences (users, then children) as one decode batch
        of logical histories; ``table`` is left empty (the block manager
        places the blocks)."""
        w = self.base
        offs = w.kv_offsets
        ks, vs, lens = [w.k], [w.v], list(w.lens)
        for i, par in enumerate(self.parents):
            lo, n = int(offs[par]), int(w.lens[par])
            ks += [w.k[lo:lo + n - 1], self.k_child[i:i + 1]]
            vs += [w.v[lo:lo + n - 1], self.v_child[i:i + 1]]
            lens.append(n)
        return Workload("prefix-forks", w.Hq, w.Hkv, w.d, w.bs, w.dtype,
                        np.asarray(lens, dtype=np.int64), np.ones(len(lens), np.int64),
                        torch.cat([w.q, self.q_child]), torch.cat(ks), torch.cat(vs),
                        np.zeros((len(lens), 0), dtype=np.int32), 0)


def prefix_fork_workload(seed=0, B=None, forks=None, device="cpu"):
    """Shared-prefix batch plus its fork step: ``forks`` parents drawn with
    numpy PCG64(seed+6) without replacement; the children's new K/V rows and
    queries from a torch generator seeded with seed+7, N(0,1) rounded to the
    config's dtype."""
    cfg = CONFIGS["prefix"]
    w = prefix_workload(seed=seed, B=B, device=device)
    nf = cfg["forks"] if forks is None else forks
    parents = np.sort(np.random.default_rng(seed + 6).choice(w.B, size=nf, replace=False))
    gen = torch.Generator().manual_seed(seed + 7)
    k_child = _values((nf, w.Hkv, w.d), w.dtype, gen, device)
    v_child = _values((nf, w.Hkv, w.d), w.dtype, gen, device)
    q_child = _values((nf, w.Hq, w.d), w.dtype, gen, device)
    return PrefixForks(w, parents, k_child, v_child, q_child)


def shared_groups_workload(groups, singles=0, seed=0, suffix_range=(1, 300), Hq=32, Hkv=8,
                           d=128, bs=16, dtype=torch.bfloat16, device="cpu"):
    """Decode batch with groups of sequences that share prefix blocks.

    groups: list of (prefix_len, members); prefix_len a multiple of bs.
    Each member's history is its group's prefix followed by a private suffix
    (uniform in suffix_range, numpy PCG64(seed)); ``singles`` more sequences
    share nothing (lengths uniform in [1, 2 * suffix_range[1]]).  The batch
    order is a seeded permutation (PCG64(seed+3)), so members of a group are
    not adjacent.  Values: torch generator seed+1, N(0,1) rounded to dtype
    (q, then per group the prefix K/V, then the private K/V of every sequence
    in batch order).  Placement: PCG64(seed+2) permutation of a pool 1.2x the
    distinct blocks; a group's prefix blocks appear once in the pool and in
    every member's table row.

    extra: shared_len [B] (the group's prefix_len for a member, else 0),
    group_start [G+1], group_seqs (batch rows of the members, group by group),
    max_group_size, max_shared_len."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lo, hi = suffix_range
    rows = []  # (group or -1, prefix_len, private_len)
    for g, (P, n) in enumerate(groups):
        assert P % bs == 0 and P > 0
        for L in rng.integers(lo, hi + 1, size=n):
            rows.append((g, P, int(L)))
    for L in rng.integers(1, 2 * hi + 1, size=singles):
        rows.append((-1, 0, int(L)))
    order = np.random.Generator(np.random.PCG64(seed + 3)).permutation(len(rows))
    rows = [rows[i] for i in order]
    B = len(rows)
    gen = torch.Generator().manual_seed(seed + 1)
    q = _values((B, Hq, d), dtype, gen, device)
    pk = [_values((P, Hkv, d), dtype, gen, device) for P, _ in groups]
    pv = [_values((P, Hkv, d), dtype, gen, device) for P, _ in groups]
    priv_k = [_values((L, Hkv, d), dtype, gen, device) for _, _, L in rows]
    priv_v = [_values((L, Hkv, d), dtype, gen, device) for _, _, L in rows]
    ks, vs, lens = [], [], []
    for (g, P, L), k_, v_ in zip(rows, priv_k, priv_v):
        ks += ([pk[g]] if g >= 0 else []) + [k_]
        vs += ([pv[g]] if g >= 0 else []) + [v_]
        lens.append(P + L)
    lens = np.asarray(lens, dtype=np.int64)
    n_pre = [P // bs for P, _ in groups]
    n_priv = [-(-L // bs) for _, _, L in rows]
    num_blocks = pool_size(n_pre + n_priv)
    perm = np.random.Generator(np.random.PCG64(seed + 2)).permutation(num_blocks)
    mb = max((P // bs if g >= 0 else 0) + -(-L // bs) for g, P, L in rows)
    table = np.zeros((B, mb), dtype=np.int32)
    pos = 0
    pre_ids = []
    for nb in n_pre:
        pre_ids.append(perm[pos:pos + nb])
        pos += nb
    for r, (g, P, L) in enumerate(rows):
        k0 = 0
        if g >= 0:
            table[r, :P // bs] = pre_ids[g]
            k0 = P // bs
        table[r, k0:k0 + n_priv[r]] = perm[pos:pos + n_priv[r]]
        pos += n_priv[r]
    shared_len = np.array([P if g >= 0 else 0 for g, P, _ in rows], dtype=np.int32)
    members = [[r for r, row in enumerate(rows) if row[0] == g] for g in range(len(groups))]
    group_start = np.concatenate([[0], np.cumsum([len(m) for m in members])]).astype(np.int32)
    group_seqs = np.array([r for m in members for r in m], dtype=np.int32)
    w = Workload("shared-groups", Hq, Hkv, d, bs, dtype, lens, np.ones(B, np.int64), q,
                 torch.cat(ks), torch.cat(vs), table, num_blocks)
    w.extra.update(shared_len=shared_len, group_start=group_start, group_seqs=group_seqs,
                   max_group_size=max((n for _, n in groups), default=0),
                   max_shared_len=max((P for P, _ in groups), default=0))
    return w


def mixed_workload(seed=0, B=None, R=None, chunk=None, priors=None, device="cpu"):
    """Continuous batch: B decode sequences plus R chunked-prefill requests.

    Returns (decode Workload, prefill Workload) sharing one pool of
    ``num_blocks`` blocks.  Prefill request r has ``extra['prior'][r]`` cached
    tokens and ``chunk`` new query tokens; its history holds prior+chunk rows.
    Priors: request 0 has 0, the last has the range maximum, the others are
    drawn uniformly in between.
    """
    cfg = CONFIGS["mixed"]
    B = B or cfg["B"]
    R = R or cfg["R"]
    n = chunk or cfg["chunk"]
    Hq, Hkv, d, bs, dtype = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["bs"], cfg["dtype"]
    rng_len = np.random.Generator(np.random.PCG64(seed))
    lo, hi = cfg["len_range"]
    lens = rng_len.integers(lo, hi + 1, size=B).astype(np.int64)
    if priors is None:
        plo, phi = cfg["prior_range"]
        mid = rng_len.integers(plo + 1, phi, size=max(R - 2, 0))
        priors = np.array([plo] + list(mid) + [phi], dtype=np.int64)[:R]
    priors = np.asarray(priors, dtype=np.int64)
    plens = priors + n
    nblk_d = _blocks_of(lens, bs)
    nblk_p = _blocks_of(plens, bs)
    num_blocks = pool_size(nblk_d + nblk_p)
    mb = max(max(nblk_d), max(nblk_p), (hi + bs - 1) // bs)
    table = place(nblk_d + nblk_p, num_blocks, np.random.Generator(np.random.PCG64(seed + 2)),
                  mb)
    gen = torch.Generator().manual_seed(seed + 1)
    qd = _values((B, Hq, d), dtype, gen, device)
    kd = _values((int(lens.sum()), Hkv, d), dtype, gen, device)
    vd = _values((int(lens.sum()), Hkv, d), dtype, gen, device)
    qp = _values((R * n, Hq, d), dtype, gen, device)
    kp = _values((int(plens.sum()), Hkv, d), dtype, gen, device)
    vp = _values((int(plens.sum()), Hkv, d), dtype, gen, device)
    dec = Workload("mixed-decode", Hq, Hkv, d, bs, dtype, lens, np.ones(B, np.int64), qd, kd, vd,
                   table[:B], num_blocks)
    pre = Workload("mixed-prefill", Hq, Hkv, d, bs, dtype, plens, np.full(R, n, np.int64), qp,
                   kp, vp, table[B:], num_blocks)
    pre.extra.update(prior=priors, chunk=n)
    return dec, pre


def sample_indices(n, k, seed=0):
    """k distinct indices of range(n), seeded, sorted."""
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    return np.sort(rng.choice(n, size=min(k, n), replace=False))
