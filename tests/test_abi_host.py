"""CPU tests of the C ABI: the library loads, exports every declared symbol, its
host generator matches the oracle bit for bit, and bad arguments are rejected
before anything is launched."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import synth
from oracle import block_pool_ref as bp
from paged_kv_cache_77_gb300 import api
from paged_kv_cache_77_gb300._lib import SIGNATURES, PagedKVError, load

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    lib = load()
    declared = _declared_symbols()
    assert len(declared) >= 15
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared <= set(SIGNATURES), declared - set(SIGNATURES)


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_generator_matches_oracle_on_workload_draws(name):
    wl = synth.WORKLOADS[name]
    d = synth.draw(wl)
    if wl.layout == "arange":
        lib_table = api.build_block_table_arange(wl.batch, d.max_blocks_per_seq)
        ref_table = bp.block_table_arange(wl.batch, d.max_blocks_per_seq)
    else:
        pool = api.BlockPool(d.num_blocks, d.pool_order)
        lib_table = pool.build_block_table(d.seq_lens, wl.block_size, wl.window, d.max_blocks_per_seq)
        rpool = bp.BlockPool(d.num_blocks, d.pool_order)
        ref_table = bp.prepare_block_tables(rpool, d.seq_lens, wl.block_size, wl.window,
                                            d.max_blocks_per_seq)
        assert pool.num_free() == rpool.num_free() and pool.null_block == rpool.null_block == 0
    assert np.array_equal(lib_table, ref_table)
    slots = api.build_slot_mapping(lib_table, d.start_pos, d.num_new, wl.block_size)
    ref_slots = bp.slot_mapping(ref_table, d.start_pos, d.num_new, wl.block_size)
    assert slots.dtype == np.int32 and np.array_equal(slots, ref_slots)
    # The same slots written into a caller's buffer (a staging buffer, say), with room
    # to spare; too small or of the wrong type is refused.
    buf = np.full(len(ref_slots) + 7, -5, dtype=np.int32)
    got = api.build_slot_mapping(lib_table, d.start_pos, d.num_new, wl.block_size, out=buf)
    assert np.array_equal(got, ref_slots) and np.shares_memory(got, buf)
    assert (buf[len(ref_slots):] == -5).all()
    for bad in (np.zeros(max(len(ref_slots) - 1, 0), np.int32), np.zeros(len(ref_slots), np.int64)):
        if len(ref_slots) == 0 and bad.dtype == np.int32:
            continue
        with pytest.raises((ValueError, PagedKVError)):
            api.build_slot_mapping(lib_table, d.start_pos, d.num_new, wl.block_size, out=bad)
    if wl.layout == "arange":
        # The pages' simplified decode formula: slot = kv_len + b * max_seq_len.
        assert np.array_equal(slots, bp.slot_mapping_contiguous_decode(
            d.start_pos, wl.max_seq_len).reshape(-1))


def test_pool_semantics_match_oracle():
    order = np.array([4, 2, 0, 3, 1, 5], dtype=np.int32)
    pool, rpool = api.BlockPool(6, order), bp.BlockPool(6, order)
    assert pool.null_block == rpool.null_block == 4
    assert pool.alloc(3).tolist() == rpool.get_new_blocks(3) == [2, 0, 3]
    pool.free([0])
    rpool.free_blocks([0])
    assert pool.alloc(3).tolist() == rpool.get_new_blocks(3) == [1, 5, 0]
    with pytest.raises(PagedKVError) as e:
        pool.alloc(1)
    assert e.value.code == -5
    for bad in ([0], [1, 1], [7]):  # null block, repeated id, out of range
        pool2 = api.BlockPool(6)
        pool2.alloc(5)
        before = pool2.num_free()
        with pytest.raises(PagedKVError) as e:
            pool2.free(bad)
        assert e.value.code == -6 and pool2.num_free() == before
    with pytest.raises(PagedKVError):
        api.BlockPool(3, np.array([0, 0, 1], dtype=np.int32))


def test_block_table_is_all_or_nothing():
    pool = api.BlockPool(10)
    with pytest.raises(PagedKVError) as e:
        pool.build_block_table([128 * 5, 128 * 5], 128, 0, 8)  # needs 10 > 9 free
    assert e.value.code == -5 and pool.num_free() == 9
    t = pool.build_block_table([128 * 5, 1], 128, 0, 8)
    assert pool.num_free() == 3 and t[1, 1:].tolist() == [0] * 7


@pytest.mark.parametrize("window", [0, 1, 100, 128, 4096])
def test_skip_count_and_sizing_match_oracle(window):
    for n in [0, 1, 99, 100, 101, 5000, 70000]:
        assert api.num_skipped_tokens(n, window) == bp.num_skipped_tokens(n, window)
    for conc, nn in [(1, 0), (7, 1), (64, 2)]:
        assert api.block_num_fixed(conc, max(window, 1), nn, 128) == bp.block_num_fixed(
            conc, max(window, 1), nn, 128)
    assert api.block_num_full_offline(2048, 128, 2) == bp.block_num_full_offline(2048, 128, 2)
    assert api.block_num_full_online(2**30, 4096, 128) == bp.block_num_full_online(2**30, 4096, 128)


def test_sliding_tables_random_lengths_match_oracle():
    rng = np.random.default_rng(11)
    for trial in range(20):
        bs = int(rng.choice([16, 128]))
        window = int(rng.integers(1, 600))
        lens = rng.integers(0, 1500, size=int(rng.integers(1, 12))).astype(np.int32)
        maxb = int(-(-lens.max() // bs)) + 1 if lens.max() > 0 else 1
        nblocks = int(sum(-(-int(n) // bs) for n in lens)) + 1
        order = np.concatenate([[0], 1 + rng.permutation(nblocks - 1)]).astype(np.int32)
        t1 = api.BlockPool(nblocks, order).build_block_table(lens, bs, window, maxb)
        t2 = bp.prepare_block_tables(bp.BlockPool(nblocks, order), lens, bs, window, maxb)
        assert np.array_equal(t1, t2)


def test_device_calls_reject_bad_arguments_before_launch():
    lib = load()
    # Unsupported head_dim: rejected before any CUDA call.
    rc = lib.pkv_paged_attention_decode(None, 1, None, None, None, None, None, 16, None, 2, 8, 2,
                                        64, 128, 10, 0.1, 0, None, 0, None, None)
    assert rc == -2
    # H not a multiple of H_kv.
    rc = lib.pkv_paged_attention_decode(None, 1, None, None, None, None, None, 16, None, 2, 9, 2,
                                        128, 128, 10, 0.1, 0, None, 0, None, None)
    assert rc == -1 and b"multiple" in lib.pkv_last_error()
    # Missing scale (non-positive) is an error, never a silent 1.0.
    rc = lib.pkv_paged_attention_decode(None, 1, None, None, None, None, None, 16, None, 2, 8, 2,
                                        128, 128, 10, 0.0, 0, None, 0, None, None)
    assert rc == -1 and b"scale" in lib.pkv_last_error()
    # Row size not a multiple of 16 bytes.
    buf = C.create_string_buffer(64)
    p = C.cast(buf, C.c_void_p)
    rc = lib.pkv_kv_cache_write(p, None, p, None, p, 1, 1, 128, 1, 3, 0, None, None)
    assert rc == -2
    # v_cache without v.
    rc = lib.pkv_kv_cache_write(p, p, p, None, p, 1, 1, 128, 1, 8, 8, None, None)
    assert rc == -1


def test_spec_decode_rejects_unsupported_shapes_before_launch():
    lib = load()
    args = lambda q_len, H, Hkv: (None, 1, None, None, None, None, None, 16, None, 2, q_len, H, Hkv,
                                  128, 128, 10, 0.1, 0, None, 0, None, None)
    # q_len outside 1..4.
    assert lib.pkv_paged_attention_decode_spec(*args(5, 8, 2)) == -2
    assert b"q_len" in lib.pkv_last_error()
    assert lib.pkv_paged_attention_decode_spec(*args(0, 8, 2)) == -2
    # More than 32 query rows per kv head: 3 tokens x 16 heads.
    assert lib.pkv_paged_attention_decode_spec(*args(3, 32, 2)) == -2
    assert b"32" in lib.pkv_last_error()
    # The workspace grows with q_len: [B*Hkv + G] slots x q_len * n_rep rows.
    one = lib.pkv_decode_spec_workspace_size(4, 1, 64, 8, 128)
    four = lib.pkv_decode_spec_workspace_size(4, 4, 64, 8, 128)
    assert one == lib.pkv_decode_workspace_size(4, 64, 8, 128) and four > 3 * one


def test_mla_spec_rejects_unsupported_shapes_before_launch():
    lib = load()
    args = lambda q_len, H, rank, scale=0.1: (None, 1, None, None, None, None, None, None, 16, None, 2,
                                              q_len, H, rank, 64, 128, 10, scale, None, 0, None, None)
    # q_len outside 1..4.
    assert lib.pkv_mla_paged_decode_spec(*args(5, 128, 512)) == -2
    assert b"q_len" in lib.pkv_last_error()
    assert lib.pkv_mla_paged_decode_spec(*args(0, 128, 512)) == -2
    # More heads than the 128-row tile, or a latent width other than 512.
    assert lib.pkv_mla_paged_decode_spec(*args(2, 129, 512)) == -2
    assert lib.pkv_mla_paged_decode_spec(*args(2, 128, 256)) == -2
    # No silent default scale.
    assert lib.pkv_mla_paged_decode_spec(*args(2, 128, 512, 0.0)) == -1
    assert b"scale" in lib.pkv_last_error()
    # Every query row is its own problem: the workspace of q_len rows over B sequences
    # is the one-row workspace of B * q_len sequences.
    assert lib.pkv_mla_decode_spec_workspace_size(4, 1, 128) == lib.pkv_mla_decode_workspace_size(4, 128)
    assert lib.pkv_mla_decode_spec_workspace_size(4, 3, 128) == lib.pkv_mla_decode_workspace_size(12, 128)
