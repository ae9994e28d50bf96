"""Pins for the oracle's host-side logic (addressing, block pool, tables, sizing).

Each pin comes from outside the oracle: the pages' worked examples (tests/golden),
brute-force enumeration, or an invariant the pages state.
"""
import json
import os

import numpy as np
import pytest

from oracle import block_pool_ref as bp

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def test_worked_slot_example():
    g = GOLD["slot_mapping_worked_example"]
    table = bp.block_table_arange(g["batch"], g["max_seq_len"] // g["block_size"])
    lb, off, pb, slot = bp.logical_to_physical(table, g["batch_idx"], g["seq_pos"], g["block_size"])
    assert (lb, off, pb, slot) == (g["logical_block"], g["offset"], g["physical_block"], g["slot"])


def test_worked_layout():
    g = GOLD["worked_layout"]
    per = g["max_seq_len"] // g["block_size"]
    assert per == g["blocks_per_seq"] and per * g["batch"] == g["total_blocks"]
    table = bp.block_table_arange(g["batch"], per)
    assert table.dtype == np.int32
    assert table[0].tolist() == g["block_table_first_row"]
    assert table[1].tolist() == g["block_table_second_row"]


def test_prefill_slot_mapping_example():
    g = GOLD["prefill_slot_mapping"]
    sm = bp.slot_mapping_contiguous_prefill(g["kv_len"], g["max_seq_len"])
    assert sm.dtype == np.int32 and len(sm) == g["length"]
    expect = np.concatenate([np.arange(a, b + 1) for a, b in g["segments"]])
    assert np.array_equal(sm, expect)
    # The general table formula gives the same slots on the arange table.
    table = bp.block_table_arange(2, g["max_seq_len"] // 128)
    gen = bp.slot_mapping(table, [0, 0], g["kv_len"], 128)
    assert np.array_equal(gen, expect)


def test_decode_slot_mapping_example():
    g = GOLD["decode_slot_mapping"]
    sm = bp.slot_mapping_contiguous_decode(g["kv_len"], g["max_seq_len"])
    assert sm.tolist() == g["slot_mapping"]
    table = bp.block_table_arange(2, g["max_seq_len"] // 128)
    gen = bp.slot_mapping(table, g["kv_len"], [1, 1], 128)
    assert gen.tolist() == [r[0] for r in g["slot_mapping"]]


def test_actual_seq_lengths_table():
    g = GOLD["actual_seq_lengths"]
    assert bp.actual_seq_lengths(g["prefill_kv_len"], "TND", "prefill").tolist() == g["tnd_prefill_kv"]
    assert bp.actual_seq_lengths(g["prefill_kv_len"], "BSH", "prefill").tolist() == g["bsh_prefill_kv"]
    assert bp.actual_seq_lengths(g["decode_kv_len"], "TND", "decode_kv").tolist() == g["tnd_decode_kv"]
    assert bp.actual_seq_lengths(g["decode_kv_len"], "TND", "decode_q").tolist() == g["tnd_decode_q"]
    assert bp.actual_seq_lengths(g["decode_kv_len"], "BSH", "decode_q").tolist() == g["bsh_decode_q"]


def test_general_formula_equals_arange_formula_everywhere():
    # The standalone guide states the two slot formulas agree when the table is arange.
    B, msl, bs = 3, 1024, 128
    table = bp.block_table_arange(B, msl // bs)
    for b in range(B):
        for pos in range(0, msl, 37):
            assert bp.logical_to_physical(table, b, pos, bs)[3] == b * msl + pos


def test_slot_inverts_to_table_entry():
    rng = np.random.default_rng(5)
    bs = 16
    table = rng.permutation(64).astype(np.int32).reshape(4, 16)
    for b in range(4):
        for pos in range(0, 256, 7):
            slot = bp.logical_to_physical(table, b, pos, bs)[3]
            assert slot // bs == table[b, pos // bs] and slot % bs == pos % bs


def test_block_pool_null_fifo_and_double_free():
    pool = bp.BlockPool(6)
    assert pool.null_block == 0 and pool.num_free() == 5
    assert pool.get_new_blocks(2) == [1, 2]
    pool.free_blocks([1])
    assert pool.get_new_blocks(3) == [3, 4, 5]
    assert pool.get_new_blocks(1) == [1]  # freed blocks go to the tail
    with pytest.raises(bp.DoubleFree):
        pool.free_blocks([0])  # the null block is never free
    pool.free_blocks([2])
    with pytest.raises(bp.DoubleFree):
        pool.free_blocks([2])
    with pytest.raises(bp.OutOfBlocks):
        pool.get_new_blocks(2)
    assert pool.num_free() == 1  # nothing was taken by the failed call


def test_block_pool_custom_order():
    pool = bp.BlockPool(5, initial_order=[3, 1, 4, 0, 2])
    assert pool.null_block == 3
    assert pool.get_new_blocks(4) == [1, 4, 0, 2]
    with pytest.raises(ValueError):
        bp.BlockPool(3, initial_order=[0, 0, 1])


@pytest.mark.parametrize("window", [1, 5, 64, 100])
def test_skip_count_matches_brute_force(window):
    for n in range(0, 300, 3):
        # n computed tokens plus the new one: visible = the newest `window` positions.
        total = n + 1
        brute = sum(1 for pos in range(total) if pos < total - window)
        assert bp.num_skipped_tokens(n, window) == brute
    assert bp.num_skipped_tokens(10**6, 0) == 0


@pytest.mark.parametrize("window", [0, 100, 128, 300])
def test_sliding_table_nulls_exactly_the_expired_blocks(window):
    bs = 32
    lens = [1, 31, 32, 33, 100, 128, 129, 300, 301, 700]
    pool = bp.BlockPool(200)
    table = bp.prepare_block_tables(pool, lens, bs, window, 25)
    seen = []
    for b, n in enumerate(lens):
        nblk = -(-n // bs)
        for j in range(25):
            if j >= nblk:
                assert table[b, j] == pool.null_block
                continue
            visible_in_block = [p for p in range(j * bs, min((j + 1) * bs, n))
                                if window == 0 or p >= n - window]
            if visible_in_block:
                assert table[b, j] != pool.null_block
                seen.append(int(table[b, j]))
            else:
                assert table[b, j] == pool.null_block
    assert len(seen) == len(set(seen))  # live blocks are distinct
    assert pool.num_free() == 199 - len(seen)


def test_blocks_to_allocate_formula_by_enumeration():
    bs = 16
    for need in range(0, 100, 5):
        for held in range(0, 8):
            blocks_covering = len({p // bs for p in range(need)})
            assert bp.num_blocks_to_allocate(need, held, bs) == max(0, blocks_covering - held)


def test_calculate_block_num_bounds():
    bs = 128
    for W in [1, 127, 128, 129, 4096]:
        for nn in [0, 1, 2]:
            L = W + 2 * nn
            worst = max(len({(off + i) // bs for i in range(L)}) for off in range(bs))
            per_req = (bp.block_num_fixed(1, W, nn, bs) - 1)
            assert per_req >= worst  # one request never spans more blocks than reserved
            assert bp.block_num_fixed(7, W, nn, bs) == 7 * per_req + 1
    assert bp.block_num_full_offline(2048, bs, 2) == 2 * 16 + 1  # worked layout + null
    assert bp.block_num_full_online(10 * 2**20, 4096, bs) == (10 * 2**20 // 4096) // bs + 1


def test_kv_len_lifecycle_drives_decode_slots():
    g = GOLD["kv_len_lifecycle"]
    kv = np.array(g["prefill"])
    table = bp.block_table_arange(2, 16)
    for step in ("after_decode_1", "after_decode_2"):
        slots = bp.slot_mapping(table, kv, [1, 1], 128)
        assert slots.tolist() == [kv[0], 2048 + kv[1]]
        kv = kv + 1
        assert kv.tolist() == g[step]
