"""Pins for the oracle's write, gather and attention (all CPU).

Each check comes from outside the oracle's own code: closed forms (one key, constant
values, zero query, two keys), positional probes that expose the visible set,
brute-force nested loops (tests/brute.py), and the equivalences the pages state
(paged = contiguous; prefill = token-by-token decode; MLA = single-head attention
with key = [nope | rope] and value = nope; GQA = repeat_kv expansion).
"""
import math

import numpy as np
import pytest

from oracle import block_pool_ref as bp
from oracle import paged_ref as ref
from tests import brute


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_bf16_widening_known_bits():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0x3E80, 0x4049], dtype=np.uint16)
    v = ref.bf16_bits_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -2.0 and v[2] == 0.0 and math.copysign(1, v[3]) < 0
    assert v[4] == math.inf and v[5] == 0.25 and v[6] == 3.140625


def test_cache_write_touches_only_target_rows():
    rng = np.random.default_rng(0)
    cache = rng.integers(0, 2**16, size=(4, 8, 2, 4), dtype=np.uint16)
    rows = rng.integers(0, 2**16, size=(3, 2, 4), dtype=np.uint16)
    slots = np.array([5, -1, 31])
    out = ref.cache_write(cache, rows, slots)
    flat_in, flat_out = cache.reshape(32, -1), out.reshape(32, -1)
    assert np.array_equal(flat_out[5], rows[0].reshape(-1))
    assert np.array_equal(flat_out[31], rows[2].reshape(-1))
    untouched = [i for i in range(32) if i not in (5, 31)]
    assert np.array_equal(flat_out[untouched], flat_in[untouched])
    assert np.array_equal(cache.reshape(32, -1), flat_in)  # input not modified
    with pytest.raises(IndexError):
        ref.cache_write(cache, rows[:1], np.array([32]))
    # No rows to write (a step with no new tokens): the cache comes back unchanged.
    empty = ref.cache_write(cache, rows[:0], np.array([], dtype=np.int64))
    assert np.array_equal(empty, cache)


def test_worked_slot_write_lands_at_block_18_offset_44():
    # The worked example: batch 1, pos 300, bs 128 on the arange table -> slot 2348.
    cache = np.zeros((32, 128, 1, 2), dtype=np.uint16)
    table = bp.block_table_arange(2, 16)
    slot = bp.logical_to_physical(table, 1, 300, 128)[3]
    out = ref.cache_write(cache, np.array([[[7, 9]]], dtype=np.uint16), np.array([slot]))
    assert out[18, 44, 0].tolist() == [7, 9] and out.sum() == 16


def test_paged_equals_contiguous_under_any_table():
    rng = np.random.default_rng(1)
    bs, Hkv, d, B = 8, 2, 4, 2
    lens = [19, 40]
    logical = [_rand(rng, n, Hkv, d) for n in lens]
    nblk = [-(-n // bs) for n in lens]
    for order in (np.arange(sum(nblk)), rng.permutation(sum(nblk))):
        cache = np.full((sum(nblk), bs, Hkv, d), np.nan)
        table = np.zeros((B, max(nblk)), dtype=np.int32)
        k = 0
        for b in range(B):
            for j in range(nblk[b]):
                table[b, j] = order[k]
                k += 1
            for pos in range(lens[b]):
                cache[table[b, pos // bs], pos % bs] = logical[b][pos]
        for b in range(B):
            assert np.array_equal(ref.gather_sequence(cache, table[b], lens[b], bs), logical[b])


def test_one_key_returns_its_value():
    rng = np.random.default_rng(2)
    q, k, v = _rand(rng, 8), _rand(rng, 1, 8), _rand(rng, 1, 5)
    o, lse, p = ref.attend(q, k, v, np.array([True]), 0.3)
    assert np.array_equal(o, v[0]) and p.tolist() == [1.0]
    assert lse == pytest.approx(0.3 * float(k[0] @ q), abs=1e-14)


def test_constant_values_and_zero_query():
    rng = np.random.default_rng(3)
    K, V = _rand(rng, 50, 16), _rand(rng, 50, 6)
    vis = np.ones(50, dtype=bool)
    o, _, p = ref.attend(_rand(rng, 16), K, np.full((50, 6), 2.5), vis, 0.25)
    assert np.allclose(o, 2.5, atol=1e-14)
    ref.check_row(o, p, np.full((50, 6), 2.5), vis)
    o, lse, _ = ref.attend(np.zeros(16), K, V, vis, 0.25)
    assert np.allclose(o, V.mean(axis=0), atol=1e-14)
    assert lse == pytest.approx(math.log(50), abs=1e-13)


def test_two_keys_sigmoid_and_scale():
    q = np.array([1.0, 0.0, 0.0])
    K = np.array([[2.0, 0.0, 0.0], [-1.0, 0.0, 0.0]])
    V = np.array([[1.0, 0.0], [0.0, 1.0]])
    scale = 0.7
    o, lse, _ = ref.attend(q, K, V, np.array([True, True]), scale)
    w1 = 1.0 / (1.0 + math.exp(-scale * 3.0))
    assert o[0] == pytest.approx(w1, abs=1e-15) and o[1] == pytest.approx(1 - w1, abs=1e-15)
    assert lse == pytest.approx(math.log(math.exp(1.4) + math.exp(-0.7)), abs=1e-14)
    # Masking the larger key leaves the other one alone.
    o, _, _ = ref.attend(q, K, V, np.array([False, True]), scale)
    assert o.tolist() == [0.0, 1.0]


def test_no_visible_key_gives_zero_and_minus_inf():
    o, lse, _ = ref.attend(np.ones(4), np.ones((3, 4)), np.ones((3, 2)), np.zeros(3, bool), 1.0)
    assert o.tolist() == [0.0, 0.0] and lse == -math.inf


def _position_valued_cache(nb, bs, Hkv, d, table, lens):
    """Cache whose value rows hold the token position, so a zero query returns the
    mean visible position."""
    v = np.full((nb, bs, Hkv, d), np.nan)
    k = np.full((nb, bs, Hkv, d), np.nan)
    for b, n in enumerate(lens):
        for pos in range(n):
            v[table[b, pos // bs], pos % bs] = pos
            k[table[b, pos // bs], pos % bs] = 1.0
    return k, v


@pytest.mark.parametrize("window", [0, 1, 7, 16, 100])
def test_decode_visible_set_by_position_probe(window):
    bs, H, d = 8, 2, 3
    lens = [1, 8, 9, 37]
    pool = bp.BlockPool(40)
    table = bp.prepare_block_tables(pool, lens, bs, window, 6)
    k, v = _position_valued_cache(40, bs, H, d, table, lens)
    o, lse = ref.paged_decode(np.zeros((4, H, d)), k, v, table, lens, bs, 0.5, window)
    for b, n in enumerate(lens):
        first = max(0, n - window) if window else 0
        assert np.allclose(o[b], (first + n - 1) / 2, atol=1e-12)
        assert np.allclose(lse[b], math.log(n - first), atol=1e-12)


def test_prefill_bottom_right_causal_by_position_probe():
    bs, H, d = 8, 1, 2
    prior, qlen = [5, 0, 20], [3, 4, 1]
    lens = [c + q for c, q in zip(prior, qlen)]
    pool = bp.BlockPool(20)
    table = bp.prepare_block_tables(pool, lens, bs, 0, 4)
    k, v = _position_valued_cache(20, bs, H, d, table, lens)
    cu = np.cumsum(qlen)
    o, _ = ref.paged_prefill(np.zeros((sum(qlen), H, d)), cu, k, v, table, lens, bs, 1.0, True)
    t = 0
    for b in range(3):
        for r in range(qlen[b]):
            assert np.allclose(o[t], (prior[b] + r) / 2, atol=1e-12)  # mean of 0..c+r
            t += 1
    o_nc, _ = ref.paged_prefill(np.zeros((sum(qlen), H, d)), cu, k, v, table, lens, bs, 1.0, False)
    assert np.allclose(o_nc[0], (lens[0] - 1) / 2)  # non-causal sees all keys
    assert not np.allclose(o_nc[0], o[0])


def test_gqa_head_mapping_matches_repeat_kv():
    # Value rows of kv head g hold g: query head h must return its kv head h // n_rep,
    # the head repeat_kv's expand(B, Hkv, n_rep, S, d).reshape(B, Hkv*n_rep, S, d) gives it.
    rng = np.random.default_rng(4)
    H, Hkv, d, bs = 8, 2, 4, 4
    lens = [9]
    table = np.array([[2, 0, 1]], dtype=np.int32)
    k = _rand(rng, 3, bs, Hkv, d)
    v = np.zeros((3, bs, Hkv, d))
    for g in range(Hkv):
        v[:, :, g, :] = g
    o, _ = ref.paged_decode(_rand(rng, 1, H, d), k, v, table, lens, bs, 0.5)
    expanded = np.repeat(np.arange(Hkv), H // Hkv)  # repeat_kv ordering
    assert np.allclose(o[0, :, 0], expanded)


def test_mha_is_gqa_with_one_query_per_kv_head():
    rng = np.random.default_rng(6)
    H, d, bs = 3, 4, 4
    lens = [10]
    table = np.array([[1, 2, 0]], dtype=np.int32)
    k, v = _rand(rng, 3, bs, H, d), _rand(rng, 3, bs, H, d)
    q = _rand(rng, 1, H, d)
    o, _ = ref.paged_decode(q, k, v, table, lens, bs, 0.5)
    for h in range(H):
        one, _ = ref.paged_decode(q[:, h:h + 1], k[:, :, h:h + 1], v[:, :, h:h + 1], table, lens, bs, 0.5)
        assert np.array_equal(o[0, h], one[0, 0])


@pytest.mark.parametrize("window", [0, 5])
def test_decode_matches_brute_force(window):
    rng = np.random.default_rng(7)
    bs, H, Hkv, d = 4, 4, 2, 3
    lens = [1, 6, 13]
    pool = bp.BlockPool(16, initial_order=[0] + list(1 + rng.permutation(15)))
    table = bp.prepare_block_tables(pool, lens, bs, window, 4)
    k, v = _rand(rng, 16, bs, Hkv, d), _rand(rng, 16, bs, Hkv, d)
    q = _rand(rng, 3, H, d)
    o, lse = ref.paged_decode(q, k, v, table, lens, bs, 0.6, window)
    for b, n in enumerate(lens):
        for h in range(H):
            kv = h // (H // Hkv)
            keys = brute.read_positions(k, table[b], n, bs, kv)
            vals = brute.read_positions(v, table[b], n, bs, kv)
            vis = [window == 0 or pos >= n - window for pos in range(n)]
            bo, blse = brute.row_attention(list(q[b, h]), keys, vals, vis, 0.6)
            assert np.allclose(o[b, h], bo, atol=1e-13) and lse[b, h] == pytest.approx(blse, abs=1e-12)


def test_prefill_matches_brute_force_and_token_by_token_decode():
    rng = np.random.default_rng(8)
    bs, H, Hkv, d = 4, 2, 1, 3
    prior, qlen = [3, 0, 9], [5, 2, 1]
    lens = [c + q for c, q in zip(prior, qlen)]
    pool = bp.BlockPool(12, initial_order=[0] + list(1 + rng.permutation(11)))
    table = bp.prepare_block_tables(pool, lens, bs, 0, 4)
    k, v = _rand(rng, 12, bs, Hkv, d), _rand(rng, 12, bs, Hkv, d)
    q = _rand(rng, sum(qlen), H, d)
    cu = np.cumsum(qlen)
    o, lse = ref.paged_prefill(q, cu, k, v, table, lens, bs, 0.4, True)
    t = 0
    for b in range(3):
        for r in range(qlen[b]):
            upto = prior[b] + r + 1
            # Row r equals a decode step that sees the first c + r + 1 keys.
            dec, dlse = ref.paged_decode(q[t:t + 1], k, v, table[b:b + 1], [upto], bs, 0.4)
            assert np.allclose(o[t], dec[0], atol=1e-14) and np.allclose(lse[t], dlse[0])
            for h in range(H):
                keys = brute.read_positions(k, table[b], lens[b], bs, 0)
                vals = brute.read_positions(v, table[b], lens[b], bs, 0)
                vis = [pos <= prior[b] + r for pos in range(lens[b])]
                bo, _ = brute.row_attention(list(q[t, h]), keys, vals, vis, 0.4)
                assert np.allclose(o[t, h], bo, atol=1e-13)
            t += 1


def test_mla_equals_single_head_attention_on_concatenated_keys():
    rng = np.random.default_rng(9)
    bs, H, dc, dr = 4, 3, 6, 2
    lens = [1, 7]
    table = np.array([[3, 0], [1, 2]], dtype=np.int32)
    nope, rope = _rand(rng, 4, bs, 1, dc), _rand(rng, 4, bs, 1, dr)
    qn, qr = _rand(rng, 2, H, dc), _rand(rng, 2, H, dr)
    o, lse = ref.mla_decode(qn, qr, nope, rope, table, lens, bs, 0.35)
    k_cat = np.concatenate([nope, rope], axis=-1)  # key = [nope | rope], value = nope
    o2, lse2 = ref.paged_decode(np.concatenate([qn, qr], axis=-1), k_cat, nope, table, lens, bs, 0.35)
    assert np.allclose(o, o2, atol=1e-14) and np.allclose(lse, lse2, atol=1e-14)
    for b, n in enumerate(lens):
        for h in range(H):
            keys = brute.read_positions(k_cat, table[b], n, bs, 0)
            vals = brute.read_positions(nope, table[b], n, bs, 0)
            bo, blse = brute.row_attention(list(np.concatenate([qn[b, h], qr[b, h]])), keys, vals,
                                           [True] * n, 0.35)
            assert np.allclose(o[b, h], bo, atol=1e-13) and lse[b, h] == pytest.approx(blse)


def test_mla_rope_term_contributes():
    # With q_nope = 0 the scores come from the rope term alone; value is still nope.
    bs = 4
    table = np.array([[0]], dtype=np.int32)
    nope = np.zeros((1, bs, 1, 2))
    nope[0, :, 0, 0] = [10.0, 20.0, 30.0, 40.0]
    rope = np.zeros((1, bs, 1, 1))
    rope[0, :, 0, 0] = [0.0, 0.0, 0.0, 50.0]
    o, _ = ref.mla_decode(np.zeros((1, 1, 2)), np.ones((1, 1, 1)), nope, rope, table, [4], bs, 1.0)
    assert o[0, 0, 0] == pytest.approx(40.0, abs=1e-12)


def test_masked_rows_never_contribute_even_if_nan():
    # The null block holds no real data; rows outside the visible set must not
    # reach the output even when they are NaN.
    rng = np.random.default_rng(12)
    K, V = _rand(rng, 6, 4), _rand(rng, 6, 3)
    K[:2] = np.nan
    V[:2] = np.nan
    vis = np.array([False, False, True, True, True, True])
    o, lse, _ = ref.attend(_rand(rng, 4), K, V, vis, 0.5)
    assert np.isfinite(o).all() and np.isfinite(lse)
    o2, lse2, _ = ref.attend(np.zeros(4), K[2:], V[2:], vis[2:], 0.5)
    o3, _, _ = ref.attend(np.zeros(4), K, V, vis, 0.5)
    assert np.allclose(o3, o2) and np.allclose(o3, V[2:].mean(axis=0))
