"""Pins for the oracle's multi-row MLA decode (several new query rows per sequence
over one latent head), all on the CPU.

Each check comes from outside that function's own code: a positional probe whose
answer is a closed form (the mean and count of the visible positions), the
reduction to the one-row MLA decode at q_len 1, the meaning of verification (row i
is the MLA decode of the prefix that ends at its own position), torch's
scaled_dot_product_attention on the concatenated [nope | rope] keys with an
explicit bottom-right mask, and nested-loop brute force.
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


def _table(rng, lens, bs, nb, max_blocks):
    pool = bp.BlockPool(nb, initial_order=[0] + list(1 + rng.permutation(nb - 1)))
    return bp.prepare_block_tables(pool, lens, bs, 0, max_blocks)


@pytest.mark.parametrize("q_len", [1, 2, 3, 4])
def test_visible_set_by_position_probe(q_len):
    rng = np.random.default_rng(70)
    bs, H, dc, dr = 4, 3, 5, 2
    lens = [0, 1, q_len, 6, 13, 30]
    B = len(lens)
    table = _table(rng, lens, bs, 40, 8)
    nope = np.zeros((40, bs, 1, dc))
    rope = _rand(rng, 40, bs, 1, dr)
    for b, n in enumerate(lens):
        for pos in range(n):
            nope[table[b, pos // bs], pos % bs, 0, 0] = pos
    # Zero queries weigh every visible row equally: column 0 of o is the mean visible
    # position and lse is log(count); a row before the sequence sees nothing.
    o, lse = ref.mla_spec_decode(np.zeros((B, q_len, H, dc)), np.zeros((B, q_len, H, dr)), nope,
                                 rope, table, lens, bs, 0.3)
    for b, n in enumerate(lens):
        for i in range(q_len):
            qpos = n - q_len + i
            if qpos < 0:
                assert np.all(o[b, i] == 0) and np.all(lse[b, i] == -np.inf)
                continue
            assert np.allclose(o[b, i, :, 0], qpos / 2, atol=1e-12)
            assert np.allclose(o[b, i, :, 1:], 0, atol=1e-12)
            assert np.allclose(lse[b, i], math.log(qpos + 1), atol=1e-12)


def test_q_len_one_is_mla_decode():
    rng = np.random.default_rng(71)
    bs, H, dc, dr = 4, 4, 6, 3
    lens = [1, 7, 14]
    table = _table(rng, lens, bs, 16, 4)
    nope, rope = _rand(rng, 16, bs, 1, dc), _rand(rng, 16, bs, 1, dr)
    qn, qr = _rand(rng, 3, H, dc), _rand(rng, 3, H, dr)
    o, lse = ref.mla_spec_decode(qn[:, None], qr[:, None], nope, rope, table, lens, bs, 0.45)
    od, lsed = ref.mla_decode(qn, qr, nope, rope, table, lens, bs, 0.45)
    assert np.array_equal(o[:, 0], od) and np.array_equal(lse[:, 0], lsed)


def test_each_row_is_the_mla_decode_of_its_prefix():
    rng = np.random.default_rng(72)
    bs, H, dc, dr, Q = 4, 3, 5, 2, 4
    lens = [4, 5, 11, 16]
    table = _table(rng, lens, bs, 20, 5)
    nope, rope = _rand(rng, 20, bs, 1, dc), _rand(rng, 20, bs, 1, dr)
    qn, qr = _rand(rng, 4, Q, H, dc), _rand(rng, 4, Q, H, dr)
    o, lse = ref.mla_spec_decode(qn, qr, nope, rope, table, lens, bs, 0.6)
    for b, n in enumerate(lens):
        for i in range(Q):
            upto = n - Q + i + 1
            od, lsed = ref.mla_decode(qn[b:b + 1, i], qr[b:b + 1, i], nope, rope, table[b:b + 1],
                                      [upto], bs, 0.6)
            assert np.allclose(o[b, i], od[0], atol=1e-14) and np.allclose(lse[b, i], lsed[0])


def test_matches_torch_sdpa_on_concatenated_keys():
    rng = np.random.default_rng(73)
    bs, H, dc, dr, Q = 8, 6, 16, 4, 3
    lens = [3, 23, 40]
    table = _table(rng, lens, bs, 24, 6)
    nope, rope = _rand(rng, 24, bs, 1, dc), _rand(rng, 24, bs, 1, dr)
    qn, qr = _rand(rng, 3, Q, H, dc), _rand(rng, 3, Q, H, dr)
    scale = 1 / math.sqrt(dc + dr)
    o, _ = ref.mla_spec_decode(qn, qr, nope, rope, table, lens, bs, scale)
    for b, n in enumerate(lens):
        rows = [table[b, pos // bs] * bs + pos % bs for pos in range(n)]
        N = torch.from_numpy(nope.reshape(-1, dc)[rows])  # [n, dc]
        R = torch.from_numpy(rope.reshape(-1, dr)[rows])
        K = torch.cat([N, R], dim=-1)[None]               # one latent head, key = [nope | rope]
        V = N[None]                                       # value = nope
        Qt = torch.from_numpy(np.concatenate([qn[b], qr[b]], axis=-1)).permute(1, 0, 2)  # [H, Q, dc+dr]
        qpos = torch.arange(n - Q, n)[:, None]
        mask = torch.arange(n)[None, :] <= qpos
        want = torch.nn.functional.scaled_dot_product_attention(
            Qt, K.expand(H, n, dc + dr), V.expand(H, n, dc), attn_mask=mask, scale=scale)
        assert np.allclose(o[b], want.permute(1, 0, 2).numpy(), atol=1e-12)


def test_matches_brute_force():
    rng = np.random.default_rng(74)
    bs, H, dc, dr, Q = 4, 2, 3, 2, 2
    lens = [1, 2, 6, 10]
    table = _table(rng, lens, bs, 16, 4)
    nope, rope = _rand(rng, 16, bs, 1, dc), _rand(rng, 16, bs, 1, dr)
    qn, qr = _rand(rng, 4, Q, H, dc), _rand(rng, 4, Q, H, dr)
    o, lse = ref.mla_spec_decode(qn, qr, nope, rope, table, lens, bs, 0.55)
    k_cat = np.concatenate([nope, rope], axis=-1)
    for b, n in enumerate(lens):
        keys = brute.read_positions(k_cat, table[b], n, bs, 0)
        vals = brute.read_positions(nope, table[b], n, bs, 0)
        for i in range(Q):
            vis = [pos <= n - Q + i for pos in range(n)]
            for h in range(H):
                qv = list(np.concatenate([qn[b, i, h], qr[b, i, h]]))
                bo, blse = brute.row_attention(qv, keys, vals, vis, 0.55)
                assert np.allclose(o[b, i, h], bo, atol=1e-13)
                if blse == -math.inf:
                    assert lse[b, i, h] == -np.inf
                else:
                    assert lse[b, i, h] == pytest.approx(blse, abs=1e-12)
