"""CPU parity of the C++ allocator (pkv_manager_*, pkv_block_hash, shared pool
blocks) with the oracle: identical block ids, reference counts and copies after
every operation of seeded random sequences."""
import random

import numpy as np
import pytest

from oracle import kv_manager_ref as km
from paged_kv_cache_77_gb300 import api
from paged_kv_cache_77_gb300._lib import PagedKVError


def _same_state(lib: api.KVCacheManager, ref: km.KVCacheManager, reqs):
    for r in reqs:
        assert lib.get_block_ids(r) == ref.get_block_ids(r), f"request {r}"
    for t, m in enumerate(ref.managers):
        assert lib.num_free(t) == m.pool.num_free()
        assert lib.null_block(t) == m.null
        for b in range(m.pool.num_blocks):
            assert lib.ref_count(t, b) == m.pool.ref[b], (t, b)
    assert lib.format_usage() == ref.format_usage()


def test_block_hash_matches_oracle_across_lengths():
    rng = np.random.default_rng(3)
    for n in list(range(0, 70)) + [128, 255, 256, 1000]:
        toks = rng.integers(-2**31, 2**31 - 1, size=n).tolist()
        for parent in (None, int(rng.integers(0, 2**63))):
            for g in (0, 1, -7):
                assert api.block_hash(parent, toks, g) == km.block_hash(parent, toks, g)


def test_pool_share_and_release_counts():
    lib = api.BlockPool(10)
    ref = km.RefBlockPool(10)
    a = lib.alloc(3).tolist()
    assert a == ref.get_new_blocks(3)
    lib.share([a[0], a[0], a[2]])
    ref.share([a[0]]); ref.share([a[0]]); ref.share([a[2]])
    for b in range(10):
        assert lib.ref_count(b) == ref.ref[b]
    lib.free([a[0], a[2], a[0]])
    ref.free_blocks([a[0], a[2], a[0]])
    with pytest.raises(PagedKVError):
        lib.free([a[1], a[1]])
    with pytest.raises(PagedKVError):
        lib.share([100])                 # out of range
    with pytest.raises(PagedKVError):
        lib.share([lib.null_block])
    for b in range(10):
        assert lib.ref_count(b) == ref.ref[b]
    assert lib.num_free() == ref.num_free()


@pytest.mark.parametrize("windows,prefix", [([0], False), ([0], True), ([24], False),
                                            ([0, 40], False), ([16, 0], False)])
def test_random_sequences_match_oracle(windows, prefix):
    seed = sum(windows) * 7 + prefix
    rng = random.Random(seed)
    nprng = np.random.default_rng(seed)
    bs, max_len = 8, 600
    nblocks = [90 + 10 * i for i in range(len(windows))]
    orders = [nprng.permutation(n).astype(np.int32) for n in nblocks]
    lib = api.KVCacheManager(windows, nblocks, bs, max_len, prefix_caching=prefix, initial_orders=orders)
    ref = km.KVCacheManager(windows, nblocks, bs, max_len, prefix_caching=prefix, initial_orders=orders)
    base = nprng.integers(0, 30, size=200).tolist()
    tokens, lens = {}, {}
    next_id = 1000
    seen = {"fork": 0, "copy": 0, "prefix_hit": 0, "full": 0, "recycled": 0}
    sw = max(range(len(windows)), key=lambda i: windows[i])  # the sliding type, if any
    for step in range(500):
        op = rng.random()
        if op < 0.35 or not lens:
            rid = next_id
            next_id += 1
            toks = base[:rng.randint(0, 120)] + nprng.integers(0, 30, size=rng.randint(1, 40)).tolist()
            cached = lib.match_prefix(rid, toks)
            assert cached == ref.match_prefix(rid, toks)
            seen["prefix_hit"] += cached > 0
            n = len(toks) - cached
            la = rng.choice([0, 0, 3])
            got = lib.allocate_slots(rid, cached, n, la)
            assert got == ref.allocate_slots(rid, cached, n, la)
            if got:
                lens[rid] = len(toks)
                tokens[rid] = toks
                lib.cache_blocks(rid, toks)
                ref.cache_blocks(rid, toks)
            else:  # a request that cannot start gives back its matched prefix
                lib.free(rid)
                ref.free(rid)
            _same_state(lib, ref, list(lens) + [rid])
        elif op < 0.65:
            rid = rng.choice(list(lens))
            k = rng.randint(1, 5)
            la = rng.choice([0, 0, 2])
            before = ref.managers[sw].pool.num_free()
            got = lib.allocate_slots(rid, lens[rid], k, la)
            assert got == ref.allocate_slots(rid, lens[rid], k, la)
            seen["full"] += not got
            seen["recycled"] += ref.managers[sw].pool.num_free() > before
            if got:
                lens[rid] += k
                tokens[rid] = tokens[rid] + nprng.integers(0, 30, size=k).tolist()
                lib.cache_blocks(rid, tokens[rid][:lens[rid]])
                ref.cache_blocks(rid, tokens[rid][:lens[rid]])
            _same_state(lib, ref, list(lens))
            continue
        elif op < 0.85:
            rid = rng.choice(list(lens))
            lib.free(rid)
            ref.free(rid)
            del lens[rid], tokens[rid]
            _same_state(lib, ref, list(lens) + [rid])
            continue
        else:
            rid = rng.choice(list(lens))
            kids = [next_id, next_id + 1]
            next_id += 2
            share = rng.random() < 0.6
            try:
                want = ref.fork(rid, kids, lens[rid], share)
            except km.OutOfBlocks:
                with pytest.raises(PagedKVError):
                    lib.fork(rid, kids, lens[rid], share)
            else:
                assert lib.fork(rid, kids, lens[rid], share) == want
                seen["fork"] += 1
                seen["copy"] += sum(len(c) for c in want)
                for kid in kids:
                    lens[kid] = lens[rid]
                    tokens[kid] = list(tokens[rid])
            _same_state(lib, ref, list(lens))
            continue
    assert seen["fork"] > 0 and seen["copy"] > 0
    assert seen["full"] > 0, "no allocation ever ran out of blocks"
    if prefix:
        assert seen["prefix_hit"] > 0
    if any(w > 0 for w in windows):
        assert seen["recycled"] > 0
