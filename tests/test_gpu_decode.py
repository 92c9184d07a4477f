"""Paged decode on the GPU against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

from gpu_util import compare, device_inputs, oracle_decode, oracle_decode_all
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


def kernel_of(w, partition_tokens=0):
    return ops().decode_kernel_for(len(w.lens), w.Hkv, w.table.shape[1], w.bs, partition_tokens)


def run(w, partition_tokens=0, seqs=None, poison=True, kernel=None):
    """Decode the batch on the GPU and the oracle; `kernel` ("persistent" or
    "grid") asserts which decode kernel the batch runs on.  With seqs=None
    every sequence is compared."""
    if kernel is not None:
        assert kernel_of(w, partition_tokens) == kernel
    k_cache, v_cache, table, lens = device_inputs(w, DEV, poison)
    out = ops().decode(w.q.to(DEV), k_cache, v_cache, table, lens,
                       partition_tokens=partition_tokens)
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    got = out.double().cpu().numpy()
    if seqs is None:
        ref = oracle_decode_all(w)
    else:
        ref = oracle_decode(w, seqs)
        got = got[np.asarray(seqs)]
    return got, ref, out


def test_tiny_fp32_config():
    """4 sequences {5,17,33,64}, MHA 4 heads, d 64, 16-token blocks, 32-block pool, fp32."""
    w = synth.decode_workload("tiny", seed=0)
    assert w.num_blocks == 32 and list(w.lens) == [5, 17, 33, 64]
    got, ref, _ = run(w, kernel="grid")
    compare(got, ref, torch.float32, "tiny")


def test_8b_config_full_size():
    """Llama-3-8B-shaped: 64 sequences, L ~ U[128,4096], 32/8 heads, d 128, bf16,
    shuffled 1.2x pool; every output element against the oracle."""
    w = synth.decode_workload("8b", seed=0)
    assert ops().decode_tile_for(w.Hq, w.Hkv, w.d, w.bs, w.num_blocks) == "tensor_core"
    got, ref, _ = run(w, kernel="persistent")
    compare(got, ref, torch.bfloat16, "8b")


def test_70b_config_full_size():
    """Llama-3-70B-shaped long context (32 sequences, L ~ U[16k,32k], 64/8
    heads, 32-token blocks, 512-token partitions): every output element of
    all 32 sequences against the oracle."""
    w = synth.decode_workload("70b", seed=0)
    assert ops().decode_tile_for(w.Hq, w.Hkv, w.d, w.bs, w.num_blocks) == "tensor_core"
    got, ref, _ = run(w, partition_tokens=512, kernel="persistent")
    compare(got, ref, torch.bfloat16, "70b")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (8, 2), (16, 2)])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_shapes_ragged(dtype, d, Hq, Hkv, bs):
    """Ragged lengths around tile, block and partition edges; 64-token
    partitions so that long sequences split and merge."""
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 300]
    w = synth.decode_workload("8b", seed=3, lens=lens, Hq=Hq, Hkv=Hkv, d=d, bs=bs, dtype=dtype,
                              max_blocks=-(-300 // bs) + 1)
    got, ref, _ = run(w, partition_tokens=max(64, bs), kernel="grid")
    compare(got, ref, dtype, f"ragged d{d} {Hq}/{Hkv} bs{bs}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (8, 2), (16, 2)])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_shapes_ragged_persistent(dtype, d, Hq, Hkv, bs):
    """The ragged lengths of test_shapes_ragged, 45 sequences with 4096-token
    tables: enough work for the persistent kernel (the 15 sequences with short
    tables above run on the grid kernel)."""
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 300] * 3
    w = synth.decode_workload("8b", seed=4, lens=lens, Hq=Hq, Hkv=Hkv, d=d, bs=bs, dtype=dtype)
    got, ref, _ = run(w, partition_tokens=max(64, bs), kernel="persistent")
    compare(got, ref, dtype, f"ragged x3 d{d} {Hq}/{Hkv} bs{bs}")


@pytest.mark.parametrize("B,kernel,Hq", [(4, "grid", 32), (64, "persistent", 32),
                                         (64, "persistent", 64)])
def test_placement_invariance_bit_identical(B, kernel, Hq):
    """Two different physical placements of the same logical K/V give
    bit-identical outputs (the reduction order follows logical positions)
    on both decode kernels and on the tensor-core tile (groups of 8)."""
    w1 = synth.decode_workload("8b", seed=5, B=B, Hq=Hq)
    w2 = synth.decode_workload("8b", seed=5, B=B, Hq=Hq)
    rng = np.random.default_rng(99)
    perm = rng.permutation(w2.num_blocks).astype(np.int32)
    w2.table = perm[w1.table]
    _, _, o1 = run(w1, seqs=[0], kernel=kernel)
    _, _, o2 = run(w2, seqs=[0])
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("B", [8, 64])
def test_split_matches_unsplit(B):
    """128- and 4096-token partitions both match the oracle (at 64 sequences
    the first runs on the persistent kernel, the second on the grid one)."""
    w = synth.decode_workload("8b", seed=6, B=B)
    _, ref, o_split = run(w, partition_tokens=128)
    _, _, o_whole = run(w, partition_tokens=4096)
    compare(o_split.double().cpu().numpy(), ref, torch.bfloat16, "split")
    compare(o_whole.double().cpu().numpy(), ref, torch.bfloat16, "whole")


@pytest.mark.parametrize("lens,Hq,Hkv,kernel", [
    ([32768], 32, 8, "grid"), ([20000, 3], 8, 1, "grid"),
    ([32768] * 9, 32, 8, "persistent"), ([20000] + [3] * 80, 8, 1, "persistent")])
def test_long_sequence_many_segments(lens, Hq, Hkv, kernel):
    """Long sequences split into 40-64 partitions of 512 tokens, merged by
    log-sum-exp: one or two sequences on the grid kernel (merge kernel over
    the partitions), and larger batches on the persistent kernel, where a
    long item spreads over more than 32 segments (the out-of-line merge)."""
    w = synth.decode_workload("8b", seed=11, lens=lens, Hq=Hq, Hkv=Hkv)
    got, ref, _ = run(w, partition_tokens=512, kernel=kernel)
    compare(got, ref, torch.bfloat16, f"long {lens}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 2)])
def test_large_batch_grid_kernel(Hq, Hkv):
    """More than 4096 sequences: the grid kernel (one CTA per sequence, KV
    head and 64-token partition) and its separate log-sum-exp merge kernel."""
    rng = np.random.default_rng(13)
    lens = [int(x) for x in rng.integers(1, 161, size=4200)]
    w = synth.decode_workload("8b", seed=13, lens=lens, Hq=Hq, Hkv=Hkv)
    got, ref, _ = run(w, partition_tokens=64, kernel="grid")
    compare(got, ref, torch.bfloat16, f"B=4200 {Hq}/{Hkv}")


@pytest.mark.parametrize("B,Hq,Hkv", [(1500, 32, 8), (3000, 8, 2), (4096, 32, 8)])
def test_large_batch_of_short_sequences_persistent(B, Hq, Hkv):
    """Up to 4096 short sequences on the persistent kernel (its [B] tables
    in shared memory: two CTAs per SM up to ~3,200 sequences, one beyond),
    with 64-token partitions so that the longer ones split; every output
    against the oracle."""
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.integers(1, 201 if B < 4096 else 121, size=B)]
    w = synth.decode_workload("8b", seed=B, lens=lens, Hq=Hq, Hkv=Hkv)
    got, ref, _ = run(w, partition_tokens=64, kernel="persistent")
    compare(got, ref, torch.bfloat16, f"B={B} {Hq}/{Hkv}")


def test_kernel_choice_follows_the_work_bound():
    """The grid kernel runs a batch while B * Hkv * partitions of the table
    capacity is at most 1.75 x the persistent grid's warps (8 per SM), and for
    B > 4096; the persistent kernel otherwise.  On a 152-SM GB300, 8B-shaped
    batches (4096-token tables, 512-token partitions) switch after 33
    sequences and 32k-token tables after 4."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for B in range(1, 200):
        for Hkv, MB, bs in ((8, 256, 16), (8, 1024, 32), (2, 64, 64)):
            parts = -(-MB * bs // 512)
            want = "grid" if 4 * B * Hkv * parts <= 7 * 8 * sms else "persistent"
            assert ops().decode_kernel_for(B, Hkv, MB, bs, 512) == want, (B, Hkv, MB, bs)
    assert ops().decode_kernel_for(4097, 8, 256, 16, 512) == "grid"
    assert ops().decode_kernel_for(4096, 8, 256, 16, 512) == "persistent"
    if sms == 152:
        assert ops().decode_kernel_for(33, 8, 256, 16, 512) == "grid"
        assert ops().decode_kernel_for(34, 8, 256, 16, 512) == "persistent"
        assert ops().decode_kernel_for(4, 8, 1024, 32, 512) == "grid"
        assert ops().decode_kernel_for(5, 8, 1024, 32, 512) == "persistent"


def test_single_token_returns_v0_exactly():
    w = synth.decode_workload("8b", seed=7, lens=[1, 1, 1])
    _, _, out = run(w)
    offs = w.kv_offsets
    g = w.Hq // w.Hkv
    for s in range(3):
        v0 = w.v[offs[s]].repeat_interleave(g, dim=0)
        assert torch.equal(out[s].cpu(), v0)


def test_zero_query_is_mean_of_values():
    w = synth.decode_workload("8b", seed=8, lens=[700, 33])
    w.q.zero_()
    got, ref, _ = run(w)
    compare(got, ref, torch.bfloat16, "q=0")
    offs = w.kv_offsets
    mean = w.v[offs[1]:offs[1] + 33].double().mean(0).repeat_interleave(4, 0).numpy()
    compare(got[1], mean, torch.bfloat16, "q=0 mean")


def test_dominant_key_selects_its_value():
    """A key with a score far above the rest (also forces the lazy rescale path
    mid-sequence)."""
    w = synth.decode_workload("8b", seed=9, lens=[1000])
    w.k[600] = w.q[0, :: w.Hq // w.Hkv].to(w.k.dtype) * 40.0
    got, ref, _ = run(w)
    compare(got, ref, torch.bfloat16, "dominant")


@pytest.mark.parametrize("nseq,kernel,Hq", [(1, "grid", 32), (64, "persistent", 32),
                                             (64, "persistent", 64)])
def test_bad_block_id_is_recorded_not_faulted(nseq, kernel, Hq):
    """An out-of-pool table entry is replaced by block 0 in the kernel and
    reported in the device error word (no out-of-bounds access), on both
    decode kernels and on the tensor-core tile (groups of 8)."""
    from paged_kv_cache_192_gb300._lib import PA_DEVERR_BAD_BLOCK
    w = synth.decode_workload("8b", seed=10, lens=[40] * nseq, Hq=Hq)
    assert kernel_of(w) == kernel
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    table[0, 1] = w.num_blocks + 5
    ops().device_error(clear=True)
    ops().decode(w.q.to(DEV), k_cache, v_cache, table, lens)
    torch.cuda.synchronize()
    assert ops().device_error(clear=True) & PA_DEVERR_BAD_BLOCK


def test_validate_mode_rejects_bad_metadata():
    from paged_kv_cache_192_gb300._lib import PAError
    w = synth.decode_workload("8b", seed=10, lens=[40, 20])
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    ops().set_validate(True)
    try:
        bad = table.clone()
        bad[1, 0] = -3
        with pytest.raises(PAError):
            ops().decode(w.q.to(DEV), k_cache, v_cache, bad, lens)
        bad_lens = lens.clone()
        bad_lens[0] = 0
        with pytest.raises(PAError):
            ops().decode(w.q.to(DEV), k_cache, v_cache, table, bad_lens)
        ops().decode(w.q.to(DEV), k_cache, v_cache, table, lens)  # valid passes
    finally:
        ops().set_validate(False)


def test_shared_prefix_equals_private_copies():
    """Sequences pointing at one physical copy of a 1024-token prefix give the
    same bits as the same sequences with private prefix copies (nalar.dev,
    'Sharing blok dapat menghindari duplikasi state KV'); both match the
    oracle."""
    w = synth.prefix_workload(seed=0, B=64)
    _, ref, o_shared = run(w, seqs=np.arange(8))
    w_priv = synth.prefix_workload(seed=0, B=64)
    w_priv.table = w_priv.extra["private_table"]
    w_priv.num_blocks = w_priv.extra["private_num_blocks"]
    _, _, o_private = run(w_priv, seqs=[0])
    assert torch.equal(o_shared, o_private)
    compare(o_shared.double().cpu().numpy()[:8], ref, torch.bfloat16, "shared prefix")


def test_prefix_config_full_size():
    """Shared-prefix config before its forks: 256 sequences, 1024 shared
    tokens, suffix ~U[1,512]; every sequence against the oracle."""
    w = synth.prefix_workload(seed=0)
    got, ref, _ = run(w)
    compare(got, ref, torch.bfloat16, "prefix")


def test_prefix_fork_step_full_size():
    """The shared-prefix config's defining step at full size: 256 users share a
    1024-token prompt (refcount 257 on its blocks), 64 of them fork a child,
    every sequence appends one token through the native block manager (parents
    whose last block is partly filled take a copy-on-write copy), then
    pa_copy_blocks, pa_reshape_and_cache of the 320 new tokens and pa_decode
    of all 320 sequences.  Each child's newest token must be in its own
    history and its parent's must not: every output against the oracle on the
    logical histories ("Apa itu PagedAttention?", section "Cara kerja
    PagedAttention", item 3; nalar.dev, section "Sharing blok dapat
    menghindari duplikasi state KV")."""
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
    n_cow = sum(1 for par in pf.parents if int(w.lens[par]) % w.bs != 0)
    assert len(st["pairs"]) == n_cow > 0
    ops().copy_blocks(k_cache, v_cache, torch.tensor(st["pairs"], dtype=torch.int64, device=DEV))
    ops().reshape_and_cache(st["k_new"].to(DEV), st["v_new"].to(DEV), k_cache, v_cache,
                            torch.from_numpy(st["new_slots"]).to(DEV))
    lw = pf.logical()
    assert np.array_equal(lw.lens, st["lens"])
    q = lw.q.to(DEV)
    table = torch.from_numpy(st["table"]).to(DEV)
    lens = torch.from_numpy(st["lens"].astype(np.int32)).to(DEV)
    out = ops().decode(q, k_cache, v_cache, table, lens)
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    compare(out.double().cpu().numpy(), oracle_decode_all(lw), torch.bfloat16, "prefix forks")
    # every prompt block is still shared by all 320 sequences (+ the prompt)
    bm = st["bm"]
    assert all(bm.refcount(b) == lw.B + 1 for b in st["table"][0, :P // w.bs])


WORKSPACE_GARBAGE_SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
from gpu_util import compare, device_inputs, oracle_decode_all
from paged_kv_cache_192_gb300 import ops, synth
w = synth.decode_workload("8b", seed=0)
assert ops.decode_kernel_for(w.B, w.Hkv, w.max_blocks, w.bs, 512) == "persistent"
k_cache, v_cache, table, lens = device_inputs(w, "cuda")
nbytes = ops.decode_workspace_size(w.B, w.Hq, w.d, w.max_blocks, w.bs, 512)
ws = torch.full((nbytes // 8,), (1 << 32) | 7, dtype=torch.int64, device="cuda")
ref = oracle_decode_all(w)
for call in range(2):
    out = ops.decode(w.q.to("cuda"), k_cache, v_cache, table, lens, partition_tokens=512,
                     workspace=ws)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    compare(out.double().cpu().numpy(), ref, torch.bfloat16, "garbage workspace call %d" % call)
    ws.fill_((1 << 32) | 7)
print("ok")
"""


def test_workspace_contents_do_not_matter_fresh_process():
    """A split batch (64 sequences of the 8B shape, items split over several
    warps) decoded in a fresh process with every workspace word set to
    (1 << 32) | 7 beforehand (stale counts and partials) still matches the
    oracle, twice: every per-item count and partial is written before it is
    read."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", WORKSPACE_GARBAGE_SCRIPT, root], cwd=root,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


@pytest.mark.parametrize("max_blocks,kernel", [(8, "grid"), (600, "persistent")])
def test_odd_query_row_count(max_blocks, kernel):
    """B x Hq odd (5 sequences x 3 query heads, 3 KV heads, d 128) with split
    sequences on both kernels: the workspace's fp32 partials stay aligned for
    the merge's vector loads whatever the number of per-item counts before
    them."""
    lens = [1, 100, 127, 128, 128] if kernel == "grid" else [1, 100, 700, 2000, 5000]
    w = synth.decode_workload("8b", seed=31, lens=lens, Hq=3, Hkv=3, max_blocks=max_blocks)
    got, ref, _ = run(w, partition_tokens=64, kernel=kernel)
    compare(got, ref, torch.bfloat16, f"odd rows {kernel}")
