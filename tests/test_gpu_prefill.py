"""Chunked prefill (causal, over paged context) on the GPU against the fp64
oracle, and the mixed continuous batch (decodes + prefill chunks)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import compare, device_inputs, oracle_decode
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


def _prefill_workload(priors, n_new, Hq=32, Hkv=8, d=128, bs=16, seed=0):
    lens = [p + n for p, n in zip(priors, n_new)]
    w = synth.decode_workload("8b", seed=seed, lens=lens, Hq=Hq, Hkv=Hkv, d=d, bs=bs)
    g = torch.Generator().manual_seed(seed + 100)
    q = torch.randn(sum(n_new), Hq, d, generator=g).to(w.dtype)
    return w, q


def _kernel(w, n_new):
    return ops().prefill_kernel_for(len(n_new), max(n_new), w.Hq, w.Hkv, w.d, w.bs,
                                    w.num_blocks, w.table.shape[1])


def _run(w, q, priors, n_new):
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    qs = torch.tensor(np.concatenate([[0], np.cumsum(n_new)]), dtype=torch.int32, device=DEV)
    out = ops().prefill_chunk(q.to(DEV), k_cache, v_cache, table, qs, lens, max(n_new))
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    ref = oracle.prefill_chunk(q.double().numpy(), w.k.double().numpy(), w.v.double().numpy(),
                               n_new, priors, 1.0 / np.sqrt(w.d))
    return out.double().cpu().numpy(), ref


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (8, 2), (32, 4)])
@pytest.mark.parametrize("d,bs", [(128, 16), (64, 32), (128, 8)])
def test_prefill_shapes(Hq, Hkv, d, bs):
    priors = [0, 13, 64, 100, 5]
    n_new = [7, 1, 65, 130, 64]
    w, q = _prefill_workload(priors, n_new, Hq, Hkv, d, bs, seed=1)
    got, ref = _run(w, q, priors, n_new)
    compare(got, ref, torch.bfloat16, f"prefill {Hq}/{Hkv} d{d} bs{bs}")


def test_prefill_many_requests_natural_order():
    """70 requests x up to 4 query tiles = 280 (request, query tile) pairs:
    past the in-kernel longest-first ranking, the pairs run in request order."""
    rng = np.random.default_rng(5)
    n_new = [int(x) for x in rng.integers(1, 201, size=70)]
    n_new[3] = 200
    priors = [int(x) for x in rng.integers(0, 300, size=70)]
    w, q = _prefill_workload(priors, n_new, Hq=8, Hkv=2, seed=5)
    assert _kernel(w, n_new) == "item_grid"
    got, ref = _run(w, q, priors, n_new)
    compare(got, ref, torch.bfloat16, "prefill 70 requests")


@pytest.mark.parametrize("Hq,Hkv,d,bs,R,nmax", [
    (32, 8, 128, 8, 30, 128),    # groups of 4: 2 query tiles of 64 tokens, 480 items
    (16, 8, 64, 16, 60, 128),    # groups of 2, head_dim 64: 480 items
    (64, 8, 128, 32, 12, 160),   # groups of 8: 32-token tiles, 5 per request, 480 items
    (8, 8, 128, 64, 60, 256),    # groups of 1: 256-token tiles, 480 items
])
def test_prefill_persistent_item_lists(Hq, Hkv, d, bs, R, nmax):
    """More work items than SMs on the persistent grid: each CTA runs a list
    of about three items (longest first to the least-loaded CTA), so the
    query-tile, K/V-ring and TMEM pipelines cross item boundaries.  Ragged
    chunks over ragged priors; every row against the oracle."""
    rng = np.random.default_rng(11 + R)
    n_new = [int(x) for x in rng.integers(1, nmax + 1, size=R)]
    n_new[0] = nmax
    priors = [int(x) for x in rng.integers(0, 700, size=R)]
    w, q = _prefill_workload(priors, n_new, Hq, Hkv, d, bs, seed=R)
    assert _kernel(w, n_new) == "persistent"
    got, ref = _run(w, q, priors, n_new)
    compare(got, ref, torch.bfloat16, f"persistent prefill {Hq}/{Hkv} d{d} bs{bs} R{R}")


@pytest.mark.parametrize("R,want", [(64, "persistent"), (65, "item_grid")])
def test_prefill_item_count_boundary(R, want):
    """64-token chunks of 32/8 heads: R requests give R x 8 work items; 512
    items still run on the persistent grid, 513+ on one CTA per item.  Both
    sides of the boundary against the oracle."""
    rng = np.random.default_rng(20 + R)
    n_new = [64] * R
    priors = [int(x) for x in rng.integers(0, 200, size=R)]
    w, q = _prefill_workload(priors, n_new, seed=R)
    assert _kernel(w, n_new) == want
    got, ref = _run(w, q, priors, n_new)
    compare(got, ref, torch.bfloat16, f"prefill {R} requests ({want})")


def test_prefill_persistent_many_one_tile_items():
    """504 one-tile items (63 requests of 1..64 new tokens, no prior context):
    each CTA runs three or four short items back to back, so every item
    boundary (query tiles reloaded, O handed over, barrier phases carried on)
    is exercised many times."""
    rng = np.random.default_rng(31)
    n_new = [int(x) for x in rng.integers(1, 65, size=63)]
    n_new[0] = 64
    priors = [0] * 63
    w, q = _prefill_workload(priors, n_new, seed=31)
    assert _kernel(w, n_new) == "persistent"
    got, ref = _run(w, q, priors, n_new)
    compare(got, ref, torch.bfloat16, "persistent prefill, 504 one-tile items")


def test_prefill_max_query_len_above_longest_chunk():
    """max_query_len larger than every request's new tokens: the extra query
    tiles have no work and the query rows' bound (R x max_query_len) exceeds
    the tokens present."""
    priors, n_new = [40, 0, 300], [17, 90, 5]
    w, q = _prefill_workload(priors, n_new, seed=13)
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    qs = torch.tensor(np.concatenate([[0], np.cumsum(n_new)]), dtype=torch.int32, device=DEV)
    assert ops().prefill_kernel_for(3, 400, w.Hq, w.Hkv, w.d, w.bs, w.num_blocks,
                                    w.table.shape[1]) == "persistent"
    out = ops().prefill_chunk(q.to(DEV), k_cache, v_cache, table, qs, lens, 400)
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    ref = oracle.prefill_chunk(q.double().numpy(), w.k.double().numpy(), w.v.double().numpy(),
                               n_new, priors, 1.0 / np.sqrt(w.d))
    compare(out.double().cpu().numpy(), ref, torch.bfloat16, "prefill, max_query_len 400")


@pytest.mark.parametrize("bs,R,want", [(16, 3, "persistent"), (16, 70, "item_grid"),
                                       (128, 3, "simple")])
def test_prefill_bad_block_id_is_recorded_not_faulted(bs, R, want):
    """An out-of-pool block-table entry of request 0 is replaced by block 0 in
    every prefill kernel and reported in the device error word (no
    out-of-bounds access); the other requests' rows still match the oracle."""
    from paged_kv_cache_192_gb300._lib import PA_DEVERR_BAD_BLOCK
    rng = np.random.default_rng(40 + R)
    n_new = [64] + [int(x) for x in rng.integers(1, 65, size=R - 1)]
    priors = [200] + [int(x) for x in rng.integers(0, 200, size=R - 1)]
    w, q = _prefill_workload(priors, n_new, Hq=8, Hkv=8, bs=bs, seed=40 + R)
    assert _kernel(w, n_new) == want
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    table[0, 1] = w.num_blocks + 5
    qs = torch.tensor(np.concatenate([[0], np.cumsum(n_new)]), dtype=torch.int32, device=DEV)
    ops().device_error(clear=True)
    out = ops().prefill_chunk(q.to(DEV), k_cache, v_cache, table, qs, lens, max(n_new))
    torch.cuda.synchronize()
    assert ops().device_error(clear=True) & PA_DEVERR_BAD_BLOCK
    ref = oracle.prefill_chunk(q.double().numpy(), w.k.double().numpy(), w.v.double().numpy(),
                               n_new, priors, 1.0 / np.sqrt(w.d))
    keep = slice(n_new[0], None)  # rows of requests 1..R-1
    compare(out.double().cpu().numpy()[keep], ref[keep], torch.bfloat16,
            f"prefill ({want}) rows beside a bad block id")


def test_prefill_persistent_one_item_per_kv_head():
    """Fewer items than SMs: one request of 3 new tokens over 61 prior ones
    gives 8 CTAs of one item each."""
    priors, n_new = [61], [3]
    w, q = _prefill_workload(priors, n_new, seed=12)
    assert _kernel(w, n_new) == "persistent"
    got, ref = _run(w, q, priors, n_new)
    compare(got, ref, torch.bfloat16, "persistent prefill, one item per KV head")


@pytest.mark.parametrize("bs", [128])
def test_prefill_large_block_fallback_kernel(bs):
    """Block size 128 is served by the 128-thread tcgen05 kernel."""
    priors = [0, 200, 77, 1000]
    n_new = [100, 129, 3, 64]
    w, q = _prefill_workload(priors, n_new, Hq=8, Hkv=2, bs=bs, seed=6)
    assert _kernel(w, n_new) == "simple"
    got, ref = _run(w, q, priors, n_new)
    compare(got, ref, torch.bfloat16, f"prefill bs{bs}")


def test_prefill_long_block_table_fallback_kernel():
    """8-token blocks over 8,300 tokens: a block table of 1,038 entries, past
    the warp-specialised kernel's staged slice."""
    priors = [8236, 5]
    n_new = [64, 40]
    w, q = _prefill_workload(priors, n_new, Hq=8, Hkv=2, bs=8, seed=7)
    assert w.table.shape[1] > 1024
    got, ref = _run(w, q, priors, n_new)
    compare(got, ref, torch.bfloat16, "prefill long table")


@pytest.mark.parametrize("bs", [16, 128])
def test_prefill_requests_without_new_tokens(bs):
    """Requests with no new tokens in the batch (n_r = 0) produce no rows and
    disturb nothing; the others match the oracle (both prefill kernels)."""
    priors = [10, 0, 3, 200, 0]
    n_new = [0, 5, 0, 70, 1]
    w, q = _prefill_workload(priors, n_new, Hq=8, Hkv=2, bs=bs, seed=9)
    got, ref = _run(w, q, priors, n_new)
    compare(got, ref, torch.bfloat16, f"prefill zero-token requests bs{bs}")


def test_prefill_first_query_sees_only_itself():
    w, q = _prefill_workload([0], [48], seed=2)
    got, _ = _run(w, q, [0], [48])
    v0 = w.v[0].repeat_interleave(w.Hq // w.Hkv, 0).double().numpy()
    assert np.array_equal(got[0], v0)


def test_mixed_config_full_size():
    """Mixed continuous batch: 128 decodes with L ~ U[256,8192] and 4 chunks of
    512 new tokens over 0..3584 prior tokens, one pool; all new K/V stored by
    reshape_and_cache first.  Every decode output and every one of the 2048
    prefill rows (all query tiles of every chunk) against the oracle."""
    from gpu_util import oracle_decode_all
    dec, pre = synth.mixed_workload(seed=0)
    from paged_kv_cache_192_gb300 import layout
    k_cache, v_cache = layout.alloc_pools(dec.num_blocks, dec.Hkv, dec.bs, dec.d, dec.dtype, DEV)
    layout.fill_pools(k_cache, v_cache, dec.k, dec.v, dec.table, dec.lens, dec.bs)
    layout.fill_pools(k_cache, v_cache, pre.k, pre.v, pre.table, pre.lens, pre.bs)
    t_dec = torch.from_numpy(dec.table).to(DEV)
    l_dec = torch.from_numpy(dec.lens.astype(np.int32)).to(DEV)
    out_d = ops().decode(dec.q.to(DEV), k_cache, v_cache, t_dec, l_dec)
    n = pre.extra["chunk"]
    R = pre.B
    qs = torch.arange(0, (R + 1) * n, n, dtype=torch.int32, device=DEV)
    assert ops().prefill_kernel_for(R, n, pre.Hq, pre.Hkv, pre.d, pre.bs, dec.num_blocks,
                                    pre.table.shape[1]) == "persistent"
    out_p = ops().prefill_chunk(pre.q.to(DEV), k_cache, v_cache, torch.from_numpy(pre.table).to(DEV),
                                qs, torch.from_numpy(pre.lens.astype(np.int32)).to(DEV), n)
    torch.cuda.synchronize()
    assert ops().device_error() == 0
    compare(out_d.double().cpu().numpy(), oracle_decode_all(dec), torch.bfloat16, "mixed decode")
    priors = pre.extra["prior"]
    ref = oracle.prefill_chunk(pre.q.double().numpy(), pre.k.double().numpy(),
                               pre.v.double().numpy(), [n] * R, priors, 1.0 / np.sqrt(pre.d))
    compare(out_p.double().cpu().numpy(), ref, torch.bfloat16, "mixed prefill (all rows)")


def test_prefill_back_to_back_calls_are_identical():
    """16 persistent-grid prefill calls issued back to back on one stream
    (each a programmatic dependent of the one before, so its set-up overlaps
    the previous call's tail) with work lists of several items per CTA: every
    output equals the first bit for bit, and the first matches the oracle."""
    rng = np.random.default_rng(77)
    R = 16  # 64 (request, query tile) pairs, at most 512 items
    n_new = [int(x) for x in rng.integers(1, 257, size=R)]
    n_new[0] = 256
    priors = [int(x) for x in rng.integers(0, 900, size=R)]
    w, q = _prefill_workload(priors, n_new, seed=77)
    assert _kernel(w, n_new) == "persistent"
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    qs = torch.tensor(np.concatenate([[0], np.cumsum(n_new)]), dtype=torch.int32, device=DEV)
    qd = q.to(DEV)
    outs = [torch.empty_like(qd) for _ in range(16)]
    ops().device_error(clear=True)
    for out in outs:
        ops().prefill_chunk(qd, k_cache, v_cache, table, qs, lens, max(n_new), out=out)
    torch.cuda.synchronize()
    assert ops().device_error(clear=True) == 0
    for i, out in enumerate(outs[1:], 1):
        assert torch.equal(out, outs[0]), f"call {i} differs from call 0"
    ref = oracle.prefill_chunk(q.double().numpy(), w.k.double().numpy(), w.v.double().numpy(),
                               n_new, priors, 1.0 / np.sqrt(w.d))
    compare(outs[0].double().cpu().numpy(), ref, torch.bfloat16, "prefill back to back")
