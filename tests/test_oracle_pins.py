"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each check is chosen so that a plausible mistake in the oracle -- a dropped
scale, a wrong softmax normalisation, an off-by-one causal mask, a wrong GQA
head map, a transposed operand, a wrong slot rule -- fails at least one of
them (the mutation tests in test_oracle_mutations.py plant such mistakes and
check exactly that).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

RNG = np.random.default_rng(1234)


def _stack(seqs):
    return np.concatenate(seqs, axis=0)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def test_two_token_closed_form_golden():
    """Hand-derived two-token case (tests/golden/closed_form_two_token.txt)."""
    exp = np.array([float(x) for x in read_golden("closed_form_two_token.txt")[0][1]])
    q = np.ones((1, 1, 4))
    k = np.array([[[1.0, 1, 1, 1]], [[0.0, 0, 0, 0]]])
    v = np.array([[[1.0, 0, 0, 0]], [[0.0, 1, 0, 0]]])
    o = oracle.decode(q, k, v, [2], 1 / math.sqrt(4), nthreads=1)
    np.testing.assert_allclose(o[0, 0], exp, rtol=0, atol=1e-15)


def test_single_token_returns_its_value():
    """L = 1: softmax over one score is 1, so o = v_0 exactly."""
    d = 8
    q = RNG.standard_normal((1, 2, d))
    k = RNG.standard_normal((1, 2, d))
    v = RNG.standard_normal((1, 2, d))
    o = oracle.decode(q, k, v, [1], 1 / math.sqrt(d), nthreads=1)
    np.testing.assert_array_equal(o[0], v[0])


def test_zero_query_is_mean_of_values():
    """q = 0: all scores 0, uniform weights, o = mean of the values."""
    L, d = 37, 16
    q = np.zeros((1, 1, d))
    k = RNG.standard_normal((L, 1, d))
    v = RNG.standard_normal((L, 1, d))
    o = oracle.decode(q, k, v, [L], 1 / math.sqrt(d), nthreads=1)
    np.testing.assert_allclose(o[0, 0], v[:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_equal_keys_is_mean_of_values():
    L, d = 19, 16
    q = RNG.standard_normal((1, 1, d))
    k = np.repeat(RNG.standard_normal((1, 1, d)), L, axis=0)
    v = RNG.standard_normal((L, 1, d))
    o = oracle.decode(q, k, v, [L], 1 / math.sqrt(d), nthreads=1)
    np.testing.assert_allclose(o[0, 0], v[:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_weights_sum_to_one():
    """All-ones values: o = sum of the softmax weights = 1."""
    L, d = 50, 32
    q = RNG.standard_normal((1, 1, d)) * 3
    k = RNG.standard_normal((L, 1, d))
    v = np.ones((L, 1, d))
    o = oracle.decode(q, k, v, [L], 1 / math.sqrt(d), nthreads=1)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value():
    """One key whose score exceeds all others by > 700: its weight is 1 to fp64
    precision, so o = v of that key (also checks the max subtraction keeps
    exp() finite for huge scores)."""
    L, d = 40, 16
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 1.0
    k = RNG.standard_normal((L, 1, d)) * 0.01
    k[23, 0, 0] = 3000.0 * math.sqrt(d)
    v = RNG.standard_normal((L, 1, d))
    o = oracle.decode(q, k, v, [L], 1 / math.sqrt(d), nthreads=1)
    np.testing.assert_allclose(o[0, 0], v[23, 0], rtol=0, atol=1e-15)


def test_gqa_head_map_contiguous_groups():
    """Hq=4, Hkv=2, L=1: query heads 0,1 read KV head 0 and heads 2,3 read KV head 1."""
    d = 4
    q = RNG.standard_normal((1, 4, d))
    k = RNG.standard_normal((1, 2, d))
    v = np.stack([np.full(d, 1.0), np.full(d, 2.0)])[None]
    o = oracle.decode(q, k, v, [1], 0.5, nthreads=1)
    np.testing.assert_array_equal(o[0, :, 0], [1.0, 1.0, 2.0, 2.0])


# --------------------------------------------------------------------------
# Against a library routine (torch scaled_dot_product_attention, float64)
# --------------------------------------------------------------------------

def _sdpa(q, k, v, mask, scale, gqa):
    """torch SDPA on [H][n][d] float64 tensors (library routine)."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(mask), scale=scale, enable_gqa=gqa).numpy()


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 4, 64), (8, 2, 32), (8, 1, 16)])
def test_decode_matches_torch_sdpa(Hq, Hkv, d):
    lens = [5, 17, 33, 64]
    q = RNG.standard_normal((len(lens), Hq, d))
    ks = [RNG.standard_normal((L, Hkv, d)) for L in lens]
    vs = [RNG.standard_normal((L, Hkv, d)) for L in lens]
    scale = 1 / math.sqrt(d)
    o = oracle.decode(q, _stack(ks), _stack(vs), lens, scale, nthreads=3)
    for s, L in enumerate(lens):
        mask = np.ones((1, L), dtype=bool)
        ref = _sdpa(q[s][:, None, :], ks[s].transpose(1, 0, 2), vs[s].transpose(1, 0, 2),
                    mask, scale, Hq != Hkv)
        np.testing.assert_allclose(o[s], ref[:, 0, :], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("prior,n", [(0, 7), (13, 9), (32, 16)])
def test_prefill_matches_torch_sdpa_causal(prior, n):
    Hq, Hkv, d = 4, 2, 16
    L = prior + n
    q = RNG.standard_normal((n, Hq, d))
    k = RNG.standard_normal((L, Hkv, d))
    v = RNG.standard_normal((L, Hkv, d))
    scale = 1 / math.sqrt(d)
    o = oracle.prefill_chunk(q, k, v, [n], [prior], scale, nthreads=2)
    # query i sits at position prior + i and sees keys 0..prior+i
    mask = np.arange(L)[None, :] <= (prior + np.arange(n))[:, None]
    ref = _sdpa(q.transpose(1, 0, 2), k.transpose(1, 0, 2), v.transpose(1, 0, 2), mask, scale,
                True)
    np.testing.assert_allclose(o, ref.transpose(1, 0, 2), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Causality and consistency
# --------------------------------------------------------------------------

def test_prefill_ignores_future_tokens():
    Hq, Hkv, d, prior, n = 2, 1, 8, 5, 6
    L = prior + n
    q = RNG.standard_normal((n, Hq, d))
    k = RNG.standard_normal((L, Hkv, d))
    v = RNG.standard_normal((L, Hkv, d))
    o1 = oracle.prefill_chunk(q, k, v, [n], [prior], 0.3, nthreads=1)
    k2, v2 = k.copy(), v.copy()
    k2[prior + 2:] += 5.0
    v2[prior + 2:] -= 7.0
    o2 = oracle.prefill_chunk(q, k2, v2, [n], [prior], 0.3, nthreads=1)
    # queries 0,1 (positions prior, prior+1) cannot see the changed rows
    np.testing.assert_array_equal(o1[:2], o2[:2])
    assert np.all(np.abs(o1[2:] - o2[2:]).max(axis=(1, 2)) > 1e-3)


def test_first_prefill_query_sees_only_itself():
    """prior = 0: query 0 sits at position 0, so its output is v_0."""
    q = RNG.standard_normal((3, 2, 8))
    k = RNG.standard_normal((3, 2, 8))
    v = RNG.standard_normal((3, 2, 8))
    o = oracle.prefill_chunk(q, k, v, [3], [0], 0.35, nthreads=1)
    np.testing.assert_array_equal(o[0], v[0])


def test_last_prefill_query_equals_decode():
    Hq, Hkv, d, prior, n = 4, 2, 16, 20, 5
    L = prior + n
    q = RNG.standard_normal((n, Hq, d))
    k = RNG.standard_normal((L, Hkv, d))
    v = RNG.standard_normal((L, Hkv, d))
    o_p = oracle.prefill_chunk(q, k, v, [n], [prior], 0.25, nthreads=1)
    o_d = oracle.decode(q[-1:], k, v, [L], 0.25, nthreads=1)
    np.testing.assert_array_equal(o_p[-1], o_d[0])


def test_thread_count_does_not_change_result():
    lens = [3, 40, 9]
    q = RNG.standard_normal((3, 4, 16))
    k = RNG.standard_normal((sum(lens), 2, 16))
    v = RNG.standard_normal((sum(lens), 2, 16))
    a = oracle.decode(q, k, v, lens, 0.25, nthreads=1)
    b = oracle.decode(q, k, v, lens, 0.25, nthreads=5)
    np.testing.assert_array_equal(a, b)


def test_bad_position_is_an_error():
    q = np.zeros((2, 1, 4))
    k = np.zeros((3, 1, 4))
    with pytest.raises(ValueError):
        oracle.attention(q, k, k, [2], [2], [3], 1.0)  # position 3 >= L = 3


# --------------------------------------------------------------------------
# Slots, scatter and block copies
# --------------------------------------------------------------------------

def test_worked_block_table_slots():
    rows = read_golden("worked_block_table.txt")
    bs = int(dict(rows)["block_size"][0])
    for tag in ("a", "b"):
        table = [int(x) for k, vals in rows if k == f"table_{tag}" for x in vals]
        for k, vals in rows:
            if k == f"slot_{tag}":
                t, expect = int(vals[0]), int(vals[1])
                got = oracle.slot_mapping(table, t + 1, bs)[t]
                assert got == expect, (tag, t, got, expect)


def test_reshape_and_cache_against_direct_indexing():
    """Brute force: every written element lands at [slot//bs, h, slot%bs, :]."""
    NB, Hkv, bs, d, T = 6, 3, 4, 5, 9
    k_new = RNG.standard_normal((T, Hkv, d)).astype(np.float32)
    v_new = RNG.standard_normal((T, Hkv, d)).astype(np.float32)
    slots = RNG.permutation(NB * bs)[:T].astype(np.int64)
    slots[3] = -1  # padding
    kc = np.full((NB, Hkv, bs, d), np.nan, np.float32)
    vc = np.full((NB, Hkv, bs, d), np.nan, np.float32)
    oracle.reshape_and_cache(k_new, v_new, kc, vc, slots, bs)
    for t in range(T):
        if slots[t] < 0:
            continue
        b, o = divmod(int(slots[t]), bs)
        for h in range(Hkv):
            np.testing.assert_array_equal(kc[b, h, o], k_new[t, h])
            np.testing.assert_array_equal(vc[b, h, o], v_new[t, h])
    written = {(int(s) // bs, int(s) % bs) for s in slots if s >= 0}
    for b in range(NB):
        for o in range(bs):
            if (b, o) not in written:
                assert np.isnan(kc[b, :, o]).all() and np.isnan(vc[b, :, o]).all()


def test_copy_blocks_copies_whole_blocks_of_both_caches():
    NB, Hkv, bs, d = 5, 2, 4, 3
    kc = RNG.standard_normal((NB, Hkv, bs, d)).astype(np.float32)
    vc = RNG.standard_normal((NB, Hkv, bs, d)).astype(np.float32)
    k0, v0 = kc.copy(), vc.copy()
    oracle.copy_blocks(kc, vc, [[1, 3], [4, 0]])
    np.testing.assert_array_equal(kc[3], k0[1])
    np.testing.assert_array_equal(vc[0], v0[4])
    for b in (1, 2, 4):
        np.testing.assert_array_equal(kc[b], k0[b])
        np.testing.assert_array_equal(vc[b], v0[b])


def test_bf16_values_upcast_exactly():
    """The oracle sees bf16 inputs exactly: bf16 -> float64 is lossless."""
    x = torch.randn(1000, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    np.testing.assert_array_equal(x.double().numpy().astype(np.float32),
                                  x.float().numpy())
