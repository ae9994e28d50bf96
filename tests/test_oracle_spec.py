"""Pins for the oracle's speculative (multi-token) decode, all on the CPU.

Each check comes from outside that function's own code: a positional probe whose
answer is a closed form (the mean and count of the visible positions), the
reduction to one-row decode at q_len 1, the meaning of verification (row i equals
the decode step of the prefix that ends at its own position), the equality with
causal prefill at a uniform q_len, nested-loop brute force, and torch's
scaled_dot_product_attention with an explicit mask.
"""
import math

import numpy as np
import pytest
import torch

from oracle import block_pool_ref as bp
from oracle import paged_ref as ref
from tests import brute


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _tables(rng, lens, bs, window, q_len, nb, max_blocks):
    # Blocks stay live from the first row's window start: the generator's window
    # is W + Q - 1 when W > 0.
    pool = bp.BlockPool(nb, initial_order=[0] + list(1 + rng.permutation(nb - 1)))
    span = window + q_len - 1 if window > 0 else 0
    return bp.prepare_block_tables(pool, lens, bs, span, max_blocks)


@pytest.mark.parametrize("window", [0, 1, 3, 9])
@pytest.mark.parametrize("q_len", [1, 2, 4])
def test_visible_set_by_position_probe(window, q_len):
    rng = np.random.default_rng(60)
    bs, H, d = 4, 2, 2
    lens = [q_len, 7, 13, 30]
    table = _tables(rng, lens, bs, window, q_len, 40, 8)
    v = np.zeros((40, bs, H, d))
    k = np.ones((40, bs, H, d))
    for b, n in enumerate(lens):
        for pos in range(n):
            v[table[b, pos // bs], pos % bs] = pos
    # A zero query weighs every visible key equally: o = mean position, lse = log(count).
    o, lse = ref.paged_spec_decode(np.zeros((4, q_len, H, d)), k, v, table, lens, bs, 0.5, window)
    for b, n in enumerate(lens):
        for i in range(q_len):
            qpos = n - q_len + i
            first = max(0, qpos - window + 1) if window else 0
            assert np.allclose(o[b, i], (first + qpos) / 2, atol=1e-12)
            assert lse[b, i] == pytest.approx(math.log(qpos - first + 1), abs=1e-12)


@pytest.mark.parametrize("window", [0, 5])
def test_q_len_one_is_decode(window):
    rng = np.random.default_rng(61)
    bs, H, Hkv, d = 4, 4, 2, 3
    lens = [1, 6, 13]
    table = _tables(rng, lens, bs, window, 1, 16, 4)
    k, v = _rand(rng, 16, bs, Hkv, d), _rand(rng, 16, bs, Hkv, d)
    q = _rand(rng, 3, H, d)
    o, lse = ref.paged_spec_decode(q[:, None], k, v, table, lens, bs, 0.6, window)
    od, lsed = ref.paged_decode(q, k, v, table, lens, bs, 0.6, window)
    assert np.array_equal(o[:, 0], od) and np.array_equal(lse[:, 0], lsed)


@pytest.mark.parametrize("window", [0, 3, 6])
def test_each_row_is_the_decode_step_of_its_prefix(window):
    rng = np.random.default_rng(62)
    bs, H, Hkv, d, Q = 4, 4, 2, 3, 3
    lens = [3, 5, 11, 16]
    table = _tables(rng, lens, bs, window, Q, 20, 5)
    k, v = _rand(rng, 20, bs, Hkv, d), _rand(rng, 20, bs, Hkv, d)
    q = _rand(rng, 4, Q, H, d)
    o, lse = ref.paged_spec_decode(q, k, v, table, lens, bs, 0.7, window)
    for b, n in enumerate(lens):
        for i in range(Q):
            upto = n - Q + i + 1
            dec, dlse = ref.paged_decode(q[b:b + 1, i], k, v, table[b:b + 1], [upto], bs, 0.7, window)
            assert np.allclose(o[b, i], dec[0], atol=1e-14) and np.allclose(lse[b, i], dlse[0])


def test_no_window_equals_causal_prefill_with_uniform_q_len():
    rng = np.random.default_rng(63)
    bs, H, Hkv, d, Q = 4, 2, 1, 3, 4
    lens = [4, 9, 17]
    table = _tables(rng, lens, bs, 0, Q, 16, 5)
    k, v = _rand(rng, 16, bs, Hkv, d), _rand(rng, 16, bs, Hkv, d)
    q = _rand(rng, 3, Q, H, d)
    o, lse = ref.paged_spec_decode(q, k, v, table, lens, bs, 0.4)
    cu = np.arange(1, 4) * Q
    op, lsep = ref.paged_prefill(q.reshape(3 * Q, H, d), cu, k, v, table, lens, bs, 0.4, True)
    assert np.allclose(o.reshape(3 * Q, H, d), op, atol=1e-14)
    assert np.allclose(lse.reshape(3 * Q, H), lsep, atol=1e-14)


@pytest.mark.parametrize("window", [0, 4])
def test_matches_brute_force(window):
    rng = np.random.default_rng(64)
    bs, H, Hkv, d, Q = 4, 4, 2, 3, 2
    lens = [2, 6, 10]
    table = _tables(rng, lens, bs, window, Q, 16, 4)
    k, v = _rand(rng, 16, bs, Hkv, d), _rand(rng, 16, bs, Hkv, d)
    q = _rand(rng, 3, Q, H, d)
    o, lse = ref.paged_spec_decode(q, k, v, table, lens, bs, 0.6, window)
    for b, n in enumerate(lens):
        for i in range(Q):
            qpos = n - Q + i
            vis = [pos <= qpos and (window == 0 or pos > qpos - window) for pos in range(n)]
            for h in range(H):
                kv = h // (H // Hkv)
                keys = brute.read_positions(k, table[b], n, bs, kv)
                vals = brute.read_positions(v, table[b], n, bs, kv)
                bo, blse = brute.row_attention(list(q[b, i, h]), keys, vals, vis, 0.6)
                assert np.allclose(o[b, i, h], bo, atol=1e-13)
                assert lse[b, i, h] == pytest.approx(blse, abs=1e-12)


def test_matches_torch_sdpa_with_explicit_mask():
    rng = np.random.default_rng(65)
    bs, H, Hkv, d, Q, W = 8, 8, 2, 16, 4, 11
    lens = [4, 23, 40]
    table = _tables(rng, lens, bs, W, Q, 24, 6)
    k, v = _rand(rng, 24, bs, Hkv, d), _rand(rng, 24, bs, Hkv, d)
    q = _rand(rng, 3, Q, H, d)
    scale = 1 / math.sqrt(d)
    o, _ = ref.paged_spec_decode(q, k, v, table, lens, bs, scale, W)
    for b, n in enumerate(lens):
        rows = [table[b, pos // bs] * bs + pos % bs for pos in range(n)]
        K = torch.from_numpy(k.reshape(-1, Hkv, d)[rows]).permute(1, 0, 2)  # [Hkv, n, d]
        V = torch.from_numpy(v.reshape(-1, Hkv, d)[rows]).permute(1, 0, 2)
        K = K.repeat_interleave(H // Hkv, dim=0)
        V = V.repeat_interleave(H // Hkv, dim=0)
        qpos = torch.arange(n - Q, n)[:, None]
        kpos = torch.arange(n)[None, :]
        mask = (kpos <= qpos) & (kpos > qpos - W)
        Qt = torch.from_numpy(q[b]).permute(1, 0, 2)  # [H, Q, d]
        want = torch.nn.functional.scaled_dot_product_attention(Qt, K, V, attn_mask=mask, scale=scale)
        assert np.allclose(o[b], want.permute(1, 0, 2).numpy(), atol=1e-12)


def test_rows_before_the_sequence_see_nothing():
    rng = np.random.default_rng(66)
    bs, H, d, Q = 4, 2, 3, 4
    lens = [2, 0]
    table = _tables(rng, lens, bs, 0, Q, 4, 2)
    k, v = _rand(rng, 4, bs, H, d), _rand(rng, 4, bs, H, d)
    q = _rand(rng, 2, Q, H, d)
    o, lse = ref.paged_spec_decode(q, k, v, table, lens, bs, 0.5)
    assert np.all(o[0, :2] == 0) and np.all(lse[0, :2] == -np.inf)
    assert np.all(np.isfinite(lse[0, 2:]))
    assert np.all(o[1] == 0) and np.all(lse[1] == -np.inf)
    # Row 2 of sequence 0 sees key 0 only, so it returns that value row.
    assert np.allclose(o[0, 2], v[table[0, 0], 0])
