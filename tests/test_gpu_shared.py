"""pa_decode_shared: groups of sequences that share prefix blocks, decoded
with the shared blocks read once per (group, KV head) and the parts merged by
log-sum-exp, against the fp64 oracle on each sequence's logical history
("PagedAttention: memetakan blok KV logis ke memori fisik tidak kontigu",
section "Sharing blok dapat menghindari duplikasi state KV")."""
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


def _groups(w):
    e = w.extra
    return (torch.from_numpy(e["shared_len"]).to(DEV), torch.from_numpy(e["group_start"]).to(DEV),
            torch.from_numpy(e["group_seqs"]).to(DEV), e["max_group_size"], e["max_shared_len"])


def run_shared(w, partition_tokens=0, kernel="persistent"):
    """pa_decode_shared and pa_decode of the batch; `kernel` asserts which
    decode kernel the batch runs on (the shared path needs the persistent
    one; None: no check)."""
    if kernel is not None:
        got = ops().decode_kernel_for(w.B, w.Hkv, w.table.shape[1], w.bs, partition_tokens)
        assert got == kernel
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    sl, gs, gm, mg, ms = _groups(w)
    out = ops().decode_shared(w.q.to(DEV), k_cache, v_cache, table, lens, sl, gs, gm, mg, ms,
                              partition_tokens=partition_tokens)
    plain = ops().decode(w.q.to(DEV), k_cache, v_cache, table, lens,
                         partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    return out, plain


@pytest.mark.parametrize("dtype_d", [128, 64])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (8, 2), (16, 2), (32, 8)])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_shared_groups_match_oracle(dtype_d, Hq, Hkv, bs):
    """Two groups (prefixes of 8 and 20 blocks, 9 and 5 members) and 120
    sequences in no group, batch order shuffled; 64-token partitions so that
    long suffixes split: every output against the oracle, and against
    pa_decode of the same batch."""
    w = synth.shared_groups_workload([(8 * bs, 9), (20 * bs, 5)], singles=120, seed=bs + Hq,
                                     Hq=Hq, Hkv=Hkv, d=dtype_d, bs=bs)
    out, plain = run_shared(w, partition_tokens=max(64, bs))
    ref = oracle_decode_all(w)
    compare(out.double().cpu().numpy(), ref, torch.bfloat16, f"shared {Hq}/{Hkv} bs{bs}")
    compare(plain.double().cpu().numpy(), ref, torch.bfloat16, "plain")


def test_shared_long_prefix_few_members_chunks():
    """A 4096-token prefix shared by 3 sequences among 30 others: the prefix
    is cut into several token chunks (one partial each) so that the prefix
    kernel has enough CTAs."""
    w = synth.shared_groups_workload([(4096, 3), (1024, 2)], singles=30, seed=5,
                                     suffix_range=(1, 700))
    out, _ = run_shared(w)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, "long prefix")


def test_shared_prefix_config_full_size():
    """Shared-prefix config (256 users x 1024 shared prompt tokens, suffix
    U[1,512]) as one group: every output against the oracle."""
    w = synth.prefix_workload(seed=0)
    B, P = w.B, w.extra["prefix"]
    w.extra.update(shared_len=np.full(B, P, np.int32), group_start=np.array([0, B], np.int32),
                   group_seqs=np.arange(B, dtype=np.int32), max_group_size=B, max_shared_len=P)
    out, _ = run_shared(w)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, "prefix shared")


def test_shared_fork_step_full_size():
    """The shared-prefix config's fork step (320 sequences after 64 forks and
    their copy-on-write copies, through the native block manager), decoded
    with the 1024-token prompt as one group of all 320: every output against
    the oracle on the logical histories."""
    from paged_kv_cache_192_gb300 import layout
    pf = synth.prefix_fork_workload(seed=0)
    w = pf.base
    st = layout.place_prefix_forks(pf, bm_seed=5)
    NB, P = st["num_blocks"], w.extra["prefix"]
    k_cache, v_cache = layout.alloc_pools(NB, w.Hkv, w.bs, w.d, w.dtype, DEV)
    ops().reshape_and_cache(w.k[:P].to(DEV), w.v[:P].to(DEV), k_cache, v_cache,
                            torch.from_numpy(st["prompt_slots"]).to(DEV))
    rows = torch.from_numpy(st["hist_rows"])
    ops().reshape_and_cache(w.k[rows].to(DEV), w.v[rows].to(DEV), k_cache, v_cache,
                            torch.from_numpy(st["hist_slots"]).to(DEV))
    ops().copy_blocks(k_cache, v_cache, torch.tensor(st["pairs"], dtype=torch.int64, device=DEV))
    ops().reshape_and_cache(st["k_new"].to(DEV), st["v_new"].to(DEV), k_cache, v_cache,
                            torch.from_numpy(st["new_slots"]).to(DEV))
    lw = pf.logical()
    B = lw.B
    table = torch.from_numpy(st["table"]).to(DEV)
    lens = torch.from_numpy(st["lens"].astype(np.int32)).to(DEV)
    sl = torch.full((B,), P, dtype=torch.int32, device=DEV)
    gs = torch.tensor([0, B], dtype=torch.int32, device=DEV)
    gm = torch.arange(B, dtype=torch.int32, device=DEV)
    ops().set_validate(True)  # the groups are consistent with the block manager's tables
    try:
        out = ops().decode_shared(lw.q.to(DEV), k_cache, v_cache, table, lens, sl, gs, gm, B, P)
    finally:
        ops().set_validate(False)
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    compare(out.double().cpu().numpy(), oracle_decode_all(lw), torch.bfloat16, "fork step shared")


def test_shared_validate_rejects_inconsistent_groups():
    from paged_kv_cache_192_gb300._lib import PAError
    w = synth.shared_groups_workload([(64, 4)], singles=40, seed=7)
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    sl, gs, gm, mg, ms = _groups(w)
    q = w.q.to(DEV)
    ops().set_validate(True)
    try:
        ops().decode_shared(q, k_cache, v_cache, table, lens, sl, gs, gm, mg, ms)  # valid
        m0, m1 = int(w.extra["group_seqs"][0]), int(w.extra["group_seqs"][1])
        bad = sl.clone()
        bad[m1] = 48  # differs inside the group
        with pytest.raises(PAError):
            ops().decode_shared(q, k_cache, v_cache, table, lens, bad, gs, gm, mg, ms)
        bad_t = table.clone()
        bad_t[m1, 0] = (int(table[m0, 0]) + 1) % w.num_blocks  # a "shared" block not shared
        with pytest.raises(PAError):
            ops().decode_shared(q, k_cache, v_cache, bad_t, lens, sl, gs, gm, mg, ms)
        two = torch.cat([gm, gm[:1]])  # a sequence in two groups
        with pytest.raises(PAError):
            ops().decode_shared(q, k_cache, v_cache, table, lens, sl,
                                torch.tensor([0, 4, 5], dtype=torch.int32, device=DEV), two, 4, ms)
    finally:
        ops().set_validate(False)


def test_shared_member_with_bad_length_is_decoded_whole():
    """Outside validate mode, a member (not the group's first) whose
    shared_len is not a multiple of the block size is decoded whole: its
    output still matches the oracle and the device error word says so."""
    from paged_kv_cache_192_gb300._lib import PA_DEVERR_BAD_BLOCK
    w = synth.shared_groups_workload([(64, 4)], singles=120, seed=8)
    assert ops().decode_kernel_for(w.B, w.Hkv, w.table.shape[1], w.bs, 64) == "persistent"
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    sl, gs, gm, mg, ms = _groups(w)
    sl[int(w.extra["group_seqs"][2])] = 40
    ops().device_error(clear=True)
    out = ops().decode_shared(w.q.to(DEV), k_cache, v_cache, table, lens, sl, gs, gm, mg, ms,
                              partition_tokens=64)
    torch.cuda.synchronize()
    assert ops().device_error(clear=True) & PA_DEVERR_BAD_BLOCK
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, "bad member")


def test_shared_small_batch_and_fp32_decode_whole():
    """Calls without the shared path (a batch small enough for the grid
    kernel; fp32) give pa_decode's result."""
    w = synth.shared_groups_workload([(64, 3)], singles=1, seed=9, suffix_range=(1, 40))
    out, plain = run_shared(w, kernel="grid")
    assert torch.equal(out, plain)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, "small")
    wf = synth.shared_groups_workload([(64, 4)], singles=120, seed=10, dtype=torch.float32)
    out, plain = run_shared(wf, partition_tokens=64)
    assert torch.equal(out, plain)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 2)])
def test_shared_groups_large_blocks_warp_level_prefix(Hq, Hkv):
    """128-token blocks: the prefix partials come from the warp-level
    tensor-core prefix kernel (the tcgen05 prefill kernel takes blocks of
    8..64 tokens); every output against the oracle."""
    w = synth.shared_groups_workload([(4 * 128, 9), (2 * 128, 5)], singles=300, seed=40 + Hq,
                                     Hq=Hq, Hkv=Hkv, bs=128)
    out, _ = run_shared(w, partition_tokens=128)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, f"bs128 {Hq}/{Hkv}")


# ---------------------------------------------------------------------------
# Forked children (pa_decode_shared_forks): the blocks a child shares with its
# parent are read once for both ("Apa itu PagedAttention?", section "Cara kerja
# PagedAttention", item 3).
# ---------------------------------------------------------------------------

def _fork(w, pairs_f):
    """Make each (child, parent, F) of pairs_f a fork: the child's first F
    tokens (logical K/V and table blocks) become the parent's."""
    offs = w.kv_offsets
    for c, par, F in pairs_f:
        assert F % w.bs == 0 and F < w.lens[c] and F < w.lens[par]
        w.k[offs[c]:offs[c] + F] = w.k[offs[par]:offs[par] + F]
        w.v[offs[c]:offs[c] + F] = w.v[offs[par]:offs[par] + F]
        w.table[c, :F // w.bs] = w.table[par, :F // w.bs]
    fp = np.full(w.B, -1, dtype=np.int32)
    fl = np.zeros(w.B, dtype=np.int32)
    for c, par, F in pairs_f:
        fp[c], fl[c] = par, F
    return torch.from_numpy(fp).to(DEV), torch.from_numpy(fl).to(DEV)


def run_forks(w, fp, fl, groups=None, partition_tokens=0, expect_error=0):
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    if groups is None:
        sl = torch.zeros(w.B, dtype=torch.int32, device=DEV)
        gs = torch.zeros(1, dtype=torch.int32, device=DEV)
        gm = torch.zeros(0, dtype=torch.int32, device=DEV)
        mg, ms = 0, 0
    else:
        sl, gs, gm, mg, ms = groups
    ops().device_error(clear=True)
    out = ops().decode_shared_forks(w.q.to(DEV), k_cache, v_cache, table, lens, sl, gs, gm, mg,
                                    ms, fp, fl, partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    assert ops().device_error(clear=True) == expect_error
    return out


def test_forks_without_groups_match_oracle():
    """64 sequences of the 8B shape, 20 of them forks of others at fork points
    from one block to nearly their whole length; no shared-prefix groups."""
    rng = np.random.default_rng(3)
    lens = [int(x) for x in rng.integers(200, 3000, size=64)]
    parents = list(range(0, 40, 2))[:20]
    children = list(range(40, 60))
    pairs = []
    for c, par in zip(children, parents):
        m = min(lens[c], lens[par]) - 1
        F = int(rng.integers(1, m // 16 + 1)) * 16
        pairs.append((c, par, F))
    w = synth.decode_workload("8b", seed=3, lens=lens)
    fp, fl = _fork(w, pairs)
    assert ops().decode_kernel_for(w.B, w.Hkv, w.table.shape[1], w.bs, 0) == "persistent"
    out = run_forks(w, fp, fl)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, "forks, no groups")


def test_forks_inside_groups_match_oracle():
    """Two prompt groups; inside each, members fork other members past the
    prompt; ungrouped sequences fork each other too."""
    w = synth.shared_groups_workload([(512, 12), (256, 10)], singles=40, seed=21,
                                     suffix_range=(40, 900))
    e = w.extra
    gs, gm, S = e["group_start"], e["group_seqs"], e["shared_len"]
    rng = np.random.default_rng(22)
    pairs = []
    for g in range(len(gs) - 1):
        mem = [int(x) for x in gm[gs[g]:gs[g + 1]]]
        for par, c in zip(mem[0::2], mem[1::2]):
            lo, hi = S[c] // w.bs, (min(w.lens[c], w.lens[par]) - 1) // w.bs
            pairs.append((c, par, int(rng.integers(lo, hi + 1)) * w.bs))
    singles = [b for b in range(w.B) if S[b] == 0]
    for par, c in zip(singles[0:20:2], singles[1:20:2]):
        hi = (min(w.lens[c], w.lens[par]) - 1) // w.bs
        pairs.append((c, par, int(rng.integers(1, hi + 1)) * w.bs))
    fp, fl = _fork(w, pairs)
    out = run_forks(w, fp, fl, groups=_groups(w), partition_tokens=64)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, "forks in groups")


def test_fork_parent_split_into_many_segments():
    """A long parent (6,000 tokens) split over many warps and 64-token
    partitions, its child forked near the end: the child gets one partial per
    segment of its parent's item (more than the merge loads speculatively)."""
    rng = np.random.default_rng(5)
    lens = [6000, 6010] + [int(x) for x in rng.integers(100, 1500, size=60)]
    w = synth.decode_workload("8b", seed=5, lens=lens)
    fp, fl = _fork(w, [(1, 0, 5984)])
    out = run_forks(w, fp, fl, partition_tokens=64)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, "long fork")


def test_two_children_of_one_parent():
    """Rows 10 and 11 both name row 3: the lower row rides with the parent, the
    other reads its fork range itself and is reported in the device error
    word; both match the oracle."""
    from paged_kv_cache_192_gb300._lib import PA_DEVERR_BAD_BLOCK
    rng = np.random.default_rng(7)
    lens = [int(x) for x in rng.integers(300, 2000, size=64)]
    lens[3], lens[10], lens[11] = 1500, 1600, 1550
    w = synth.decode_workload("8b", seed=7, lens=lens)
    fp, fl = _fork(w, [(10, 3, 800), (11, 3, 1200)])
    out = run_forks(w, fp, fl, expect_error=PA_DEVERR_BAD_BLOCK)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, "two children")


@pytest.mark.parametrize("bad", ["len", "beyond", "chain"])
def test_invalid_fork_is_recorded_and_read_whole(bad):
    """A fork length that is no multiple of the block size, one at the
    child's length, or a parent that is itself a child: the child reads its
    whole range, the error is recorded, every output still matches."""
    from paged_kv_cache_192_gb300._lib import PA_DEVERR_BAD_BLOCK
    rng = np.random.default_rng(9)
    lens = [int(x) for x in rng.integers(300, 2000, size=64)]
    lens[5], lens[6], lens[7] = 1000, 1000, 1000
    w = synth.decode_workload("8b", seed=9, lens=lens)
    fp, fl = _fork(w, [(6, 5, 480), (7, 6, 320)] if bad == "chain" else [(6, 5, 480)])
    if bad == "len":
        fl[6] = 479
    elif bad == "beyond":
        fl[6] = 1008
    out = run_forks(w, fp, fl, expect_error=PA_DEVERR_BAD_BLOCK)
    compare(out.double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16, f"bad fork {bad}")


def test_fork_validate_mode_rejects_bad_forks():
    from paged_kv_cache_192_gb300._lib import PAError
    rng = np.random.default_rng(11)
    lens = [int(x) for x in rng.integers(300, 2000, size=48)]
    w = synth.decode_workload("8b", seed=11, lens=lens)
    fp, fl = _fork(w, [(6, 5, 160)])
    k_cache, v_cache, table, lens_d = device_inputs(w, DEV)
    sl = torch.zeros(w.B, dtype=torch.int32, device=DEV)
    gs = torch.zeros(1, dtype=torch.int32, device=DEV)
    gm = torch.zeros(0, dtype=torch.int32, device=DEV)
    table[6, 2] = table[6, 2] + 1  # the rows now differ before the fork
    ops().set_validate(True)
    try:
        with pytest.raises(PAError):
            ops().decode_shared_forks(w.q.to(DEV), k_cache, v_cache, table, lens_d, sl, gs, gm,
                                      0, 0, fp, fl)
    finally:
        ops().set_validate(False)


def test_prefix_fork_step_with_forks_full_size():
    """The shared-prefix config's fork step (256 users sharing a 1024-token
    prompt, 64 forks, copy-on-write, 320 new tokens) decoded with the prompt
    group and the 64 forks: each child's blocks before its parent's last,
    partly filled one are read once for both; every output against the
    oracle."""
    from paged_kv_cache_192_gb300 import layout
    pf = synth.prefix_fork_workload(seed=0)
    w = pf.base
    st = layout.place_prefix_forks(pf, bm_seed=5)
    NB, P, bs = st["num_blocks"], w.extra["prefix"], w.bs
    k_cache, v_cache = layout.alloc_pools(NB, w.Hkv, w.bs, w.d, w.dtype, DEV)
    ops().reshape_and_cache(w.k[:P].to(DEV), w.v[:P].to(DEV), k_cache, v_cache,
                            torch.from_numpy(st["prompt_slots"]).to(DEV))
    rows = torch.from_numpy(st["hist_rows"])
    ops().reshape_and_cache(w.k[rows].to(DEV), w.v[rows].to(DEV), k_cache, v_cache,
                            torch.from_numpy(st["hist_slots"]).to(DEV))
    ops().copy_blocks(k_cache, v_cache, torch.tensor(st["pairs"], dtype=torch.int64, device=DEV))
    ops().reshape_and_cache(st["k_new"].to(DEV), st["v_new"].to(DEV), k_cache, v_cache,
                            torch.from_numpy(st["new_slots"]).to(DEV))
    lw = pf.logical()
    Bt = lw.B
    fp = np.full(Bt, -1, dtype=np.int32)
    fl = np.zeros(Bt, dtype=np.int32)
    for i, par in enumerate(pf.parents):
        c = w.B + i
        fp[c], fl[c] = par, (int(w.lens[par]) - 1) // bs * bs
        assert np.array_equal(st["table"][c, :fl[c] // bs], st["table"][par, :fl[c] // bs])
    table = torch.from_numpy(st["table"]).to(DEV)
    lens = torch.from_numpy(st["lens"].astype(np.int32)).to(DEV)
    sl = torch.full((Bt,), P, dtype=torch.int32, device=DEV)
    gs = torch.tensor([0, Bt], dtype=torch.int32, device=DEV)
    gm = torch.arange(Bt, dtype=torch.int32, device=DEV)
    ops().device_error(clear=True)
    out = ops().decode_shared_forks(lw.q.to(DEV), k_cache, v_cache, table, lens, sl, gs, gm, Bt, P,
                                    torch.from_numpy(fp).to(DEV), torch.from_numpy(fl).to(DEV))
    torch.cuda.synchronize()
    assert ops().device_error(clear=True) == 0
    compare(out.double().cpu().numpy(), oracle_decode_all(lw), torch.bfloat16, "fork step, forks")


@pytest.mark.parametrize("forks", [False, True])
def test_back_to_back_calls_are_identical(forks):
    """24 calls issued back to back on one stream with one workspace and no
    synchronisation between them: each call's decode grid releases the
    shared-prefix kernel at its start and that kernel releases the merge, so
    consecutive calls overlap their launches; every output must equal the
    first bit for bit, and the first must match the oracle."""
    w = synth.shared_groups_workload([(512, 12), (256, 10)], singles=40, seed=31,
                                     suffix_range=(40, 900))
    fp = fl = None
    if forks:
        S = w.extra["shared_len"]
        singles = [b for b in range(w.B) if S[b] == 0]
        pairs = []
        for par, c in zip(singles[0:16:2], singles[1:16:2]):
            hi = (min(w.lens[c], w.lens[par]) - 1) // w.bs
            if hi > 0:  # a fork shares at least one whole block
                pairs.append((c, par, hi * w.bs))
        assert len(pairs) >= 6
        fp, fl = _fork(w, pairs)
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    sl, gs, gm, mg, ms = _groups(w)
    q = w.q.to(DEV)
    MB = table.shape[1]
    wsf = ops().decode_shared_forks_workspace_size if forks else ops().decode_shared_workspace_size
    ws = torch.empty(wsf(w.B, w.Hq, w.d, MB, w.bs, 64, ms) // 4, dtype=torch.float32, device=DEV)
    outs = [torch.empty_like(q) for _ in range(24)]
    ops().device_error(clear=True)
    for out in outs:
        if forks:
            ops().decode_shared_forks(q, k_cache, v_cache, table, lens, sl, gs, gm, mg, ms, fp, fl,
                                      partition_tokens=64, workspace=ws, out=out)
        else:
            ops().decode_shared(q, k_cache, v_cache, table, lens, sl, gs, gm, mg, ms,
                                partition_tokens=64, workspace=ws, out=out)
    torch.cuda.synchronize()
    assert ops().device_error(clear=True) == 0
    for i, out in enumerate(outs[1:], 1):
        assert torch.equal(out, outs[0]), f"call {i} differs from call 0"
    compare(outs[0].double().cpu().numpy(), oracle_decode_all(w), torch.bfloat16,
            "back to back" + (" with forks" if forks else ""))
