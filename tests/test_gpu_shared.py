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
