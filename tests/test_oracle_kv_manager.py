"""Pins of the allocator oracle (oracle/kv_manager_ref.py) against the pages and
against properties that enumeration can check, independent of its formulas."""
import json
import os
import random
import subprocess
import sys

import numpy as np
import pytest

from oracle import kv_manager_ref as km

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def _invariants(mgr: km.KVCacheManager):
    """Reference counts equal the holdings; the queue holds exactly the unheld ids."""
    for m in mgr.managers:
        held = {}
        for blocks in m.req_to_blocks.values():
            for b in blocks:
                if b != m.null:
                    held[b] = held.get(b, 0) + 1
        q = list(m.pool.queue)
        assert len(q) == len(set(q)), "duplicate id in the free queue"
        assert m.null not in q
        for b in range(m.pool.num_blocks):
            assert m.pool.ref[b] == held.get(b, 0), f"block {b}: ref {m.pool.ref[b]} held {held.get(b, 0)}"
            if b != m.null:
                assert (b in q) == (held.get(b, 0) == 0)
        for h, b in m.hash_to_block.items():
            assert m.block_to_hash[b] == h and m.pool.ref[b] > 0


def test_blocks_to_allocate_formula_from_page():
    # Full attention: the printed formula, through the manager's own counting.
    for c in GOLD["blocks_to_allocate_formula"]["cases"]:
        pool = km.RefBlockPool(64)
        m = km.SingleTypeManager(pool, c["block_size"], 1 << 20)
        m.req_to_blocks[7] = pool.get_new_blocks(c["existing"])
        assert m.get_num_blocks_to_allocate(7, c["num_tokens_need_slot"], 0) == c["allocate"]


def test_fork_example_from_page():
    g = GOLD["fork_blocks_example"]
    bs = 16
    num_tokens = (g["parent_blocks"] - 1) * bs + 5  # last block incomplete
    for shareable in (False, True):
        mgr = km.KVCacheManager([0], [64], bs, 4096)
        assert mgr.allocate_slots(1, 0, num_tokens)
        parent = mgr.get_block_ids(1)[0]
        assert len(parent) == g["parent_blocks"]
        free0 = mgr.managers[0].pool.num_free()
        copies = mgr.fork(1, [2, 3], num_tokens, shareable)[0]
        new = free0 - mgr.managers[0].pool.num_free()
        if shareable:
            assert new == g["shared_new_blocks"] and len(copies) == g["shared_new_blocks"]
            for b in parent[:-1]:
                assert mgr.managers[0].pool.ref[b] == 1 + g["shared_full_block_ref_increment"]
            assert all(s == parent[-1] for s, _ in copies)
        else:
            assert new == g["unshared_new_blocks"] and len(copies) == g["unshared_copies"]
            assert all(mgr.managers[0].pool.ref[b] == 1 for b in parent)
        for child in (2, 3):
            row = mgr.get_block_ids(child)[0]
            assert len(row) == g["parent_blocks"]
        _invariants(mgr)
        # Freeing the parent keeps shared blocks alive for the children.
        mgr.free(1)
        _invariants(mgr)
        mgr.free(2)
        mgr.free(3)
        assert mgr.managers[0].pool.num_free() == 63
        _invariants(mgr)


def test_format_usage_example_from_page():
    g = GOLD["format_usage_example"]
    # Block size 1, window 9: after 12 computed tokens the next query sees
    # positions 4..12, so the sliding list keeps 8 of its 12 blocks.
    mgr = km.KVCacheManager([0, 9], [g["full"]["total"], g["sliding"]["total"]], 1, 1 << 20)
    assert mgr.allocate_slots(5, 0, 12)
    assert mgr.allocate_slots(5, 12, 0)
    m_sl = mgr.managers[1]
    assert sum(b != m_sl.null for b in mgr.get_block_ids(5)[1]) == 8
    assert mgr.format_usage() == g["text"]


def test_full_attention_decode_growth_by_enumeration():
    bs = 8
    mgr = km.KVCacheManager([0], [200], bs, 10_000)
    assert mgr.allocate_slots(0, 0, 5)
    n = 5
    for _ in range(300):
        assert mgr.allocate_slots(0, n, 1)
        n += 1
        row = mgr.get_block_ids(0)[0]
        assert len(row) == len({p // bs for p in range(n)})
        assert len(set(row)) == len(row) and mgr.managers[0].null not in row
    _invariants(mgr)


@pytest.mark.parametrize("W,bs", [(16, 4), (33, 8), (128, 128), (5, 16)])
def test_sliding_window_positions_backed(W, bs):
    rng = random.Random(W * 131 + bs)
    mgr = km.KVCacheManager([W], [400], bs, 100_000)
    m = mgr.managers[0]
    c = 0
    for step in range(200):
        n = rng.choice([1, 1, 1, 2, 3, 7, 20, 50])
        la = rng.choice([0, 0, 2])
        assert mgr.allocate_slots(9, c, n, la)
        row = mgr.get_block_ids(9)[0]
        need = c + n + la
        first_visible = max(0, c - W + 1)  # the first new query sees from here
        for p in range(first_visible, need):
            assert row[p // bs] != m.null, (step, p)
        for j, b in enumerate(row):
            if (j + 1) * bs <= first_visible:
                assert b == m.null, (step, j)
        c += n
        _invariants(mgr)
    # The real blocks never exceed what the window and one step need.
    assert sum(b != m.null for b in row) <= km.ceil_div(W - 1 + 50 + 2, bs) + 1


def test_two_phase_is_all_or_nothing():
    mgr = km.KVCacheManager([0, 64], [1000, 6], 16, 1 << 20)
    assert mgr.allocate_slots(1, 0, 40)          # full 3 blocks, sliding 3 blocks
    before = mgr.get_block_ids(1)
    free_full = mgr.managers[0].pool.num_free()
    # 200 more tokens: the sliding pool (2 free) cannot cover the window layout.
    assert not mgr.allocate_slots(2, 0, 200)
    assert mgr.get_block_ids(2) == [[], []]
    assert mgr.managers[0].pool.num_free() == free_full
    assert mgr.get_block_ids(1) == before
    _invariants(mgr)


def test_release_more_than_referenced_is_double_free():
    pool = km.RefBlockPool(8)
    a = pool.get_new_blocks(2)
    pool.share([a[0]])
    pool.free_blocks([a[0], a[0]])           # two references, two releases: fine
    with pytest.raises(km.DoubleFree):
        pool.free_blocks([a[0]])
    with pytest.raises(km.DoubleFree):
        pool.free_blocks([a[1], a[1]])
    with pytest.raises(km.DoubleFree):
        pool.free_blocks([pool.null_block])


def test_blake2b_is_the_rfc_function():
    # RFC 7693 Appendix A: BLAKE2b-512("abc").
    assert hashlib_hex(b"abc") == (
        "ba80a53f981c4d0d6a2797b69f12f6e94c212f14685ac4b74b12bb6fdbffa2d1"
        "7d87c5392aab792dc252d5de4533cc9518d38aa8dbf1925ab92386edd4009923")


def hashlib_hex(data):
    import hashlib
    return hashlib.blake2b(data).hexdigest()


def test_block_hash_is_process_independent():
    # The page's warning: Python's hash() is salted per process; the fingerprint
    # must be the same in every process (tensor-parallel ranks).
    toks = list(range(100, 116))
    here = km.block_hash(None, toks, 0), km.block_hash(12345, toks, 1)
    code = ("from oracle import kv_manager_ref as km; "
            "print(km.block_hash(None, list(range(100, 116)), 0), km.block_hash(12345, list(range(100, 116)), 1))")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, check=True,
                         env={**os.environ, "PYTHONHASHSEED": "977"},
                         cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert tuple(int(x) for x in out.stdout.split()) == here
    # Parent, tokens and group each change the fingerprint.
    assert len({km.block_hash(None, toks, 0), km.block_hash(1, toks, 0),
                km.block_hash(None, toks[:-1] + [0], 0), km.block_hash(None, toks, 1)}) == 4


def test_prefix_match_against_token_comparison():
    # Brute force: a prefix of j full blocks is shared when some live request that
    # fingerprinted them holds exactly those tokens in its first j blocks.
    rng = np.random.default_rng(5)
    bs = 4
    mgr = km.KVCacheManager([0], [300], bs, 1 << 20, prefix_caching=True)
    base = rng.integers(0, 50, size=64).tolist()
    live = {}
    for rid in range(40):
        cut = int(rng.integers(0, 64))
        toks = base[:cut] + rng.integers(0, 50, size=int(rng.integers(1, 20))).tolist()
        # Brute-force expectation over live requests.
        limit = (len(toks) - 1) // bs
        expect = 0
        m = mgr.managers[0]
        for orid, other in live.items():
            # Only fingerprinted blocks can be shared: a block whose content was
            # computed a second time (its fingerprint already taken) is not.
            row = m.req_to_blocks[orid]
            n = 0
            while (n < min(limit, len(other) // bs) and row[n] in m.block_to_hash
                   and other[n * bs:(n + 1) * bs] == toks[n * bs:(n + 1) * bs]):
                n += 1
            expect = max(expect, n)
        cached = mgr.match_prefix(rid, toks)
        assert cached == expect * bs, (rid, cached, expect)
        assert mgr.allocate_slots(rid, cached, len(toks) - cached)
        mgr.cache_blocks(rid, toks)
        live[rid] = toks
        _invariants(mgr)
        if rng.random() < 0.3:
            victim = int(rng.choice(list(live)))
            mgr.free(victim)
            del live[victim]
            _invariants(mgr)


def test_random_operations_keep_invariants():
    rng = random.Random(11)
    mgr = km.KVCacheManager([0, 24], [120, 60], 8, 4000, prefix_caching=False)
    lens = {}
    next_id = 0
    for _ in range(600):
        op = rng.random()
        if op < 0.45 or not lens:
            rid = next_id
            next_id += 1
            n = rng.randint(1, 60)
            if mgr.allocate_slots(rid, 0, n):
                lens[rid] = n
        elif op < 0.75:
            rid = rng.choice(list(lens))
            k = rng.randint(1, 4)
            if mgr.allocate_slots(rid, lens[rid], k):
                lens[rid] += k
        elif op < 0.9:
            rid = rng.choice(list(lens))
            mgr.free(rid)
            del lens[rid]
        else:
            rid = rng.choice(list(lens))
            kids = [next_id, next_id + 1]
            next_id += 2
            try:
                mgr.fork(rid, kids, lens[rid], shareable=rng.random() < 0.5)
                for kid in kids:
                    lens[kid] = lens[rid]
            except km.OutOfBlocks:
                pass
        _invariants(mgr)
