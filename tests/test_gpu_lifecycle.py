"""GPU parity over a continuous-batching run: a few hundred decode steps driven by the
library's own allocator, replayed step by step by the oracle.

Two attention types share one request set, as in a model with full-attention and
sliding-window layers ("KV Cache 管理设计文档" §2.2-§2.3: one single-type manager and
one block pool per type; §3 allocate_slots in two phases). Each step, for every live
request, the library's manager grows the block lists by one token
(pkv_manager_allocate_slots with computed = kv_len, one new token), which for the
sliding type first recycles the blocks that left the window to the pool
(remove_skipped_blocks, §2.3.2); the C generator turns the tables into slots; the
new K/V row of every request is written into each type's cache; then each type's
cache is decoded (full attention, and the window). kv_len grows by one after the
step ("KVCache 优化技能" §3.5, the life of kv_len). Along the way a request forks
into two children that decode on divergent tokens, one request finishes and frees
its blocks, and a new request is admitted with a prompt that lands in recycled
blocks.

At every step: the library's block lists and tables equal the oracle manager's, the
caches after the write equal the oracle's write bit for bit, and the decode outputs
match the oracle within the decode tolerance.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import block_pool_ref as bp
from oracle import kv_manager_ref as km
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import compare

pytestmark = pytest.mark.gpu

BS, HKV, D, H = 128, 2, 128, 8
WINDOW = 160          # sliding type: the window passes a block boundary every 128 steps
MAXB = 8              # max blocks per sequence (1024 tokens)
STEPS = 300
FORK_AT, SWAP_AT = 100, 150


def _rand_bf16(shape, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


class Layer:
    """One attention type: its GPU caches and the oracle's bit copies."""

    def __init__(self, nb, gen, window):
        self.window = window
        self.k = _rand_bf16((nb, BS, HKV, D), gen).cuda()
        self.v = _rand_bf16((nb, BS, HKV, D), gen).cuda()
        self.kc, self.vc = synth.bf16_bits(self.k), synth.bf16_bits(self.v)

    def write(self, slots, k_rows, v_rows, status):
        api.kv_cache_write(self.k, self.v, k_rows.cuda(), v_rows.cuda(),
                           torch.from_numpy(slots).cuda(), dev_status=status)
        self.kc = ref.cache_write(self.kc, synth.bf16_bits(k_rows), slots)
        self.vc = ref.cache_write(self.vc, synth.bf16_bits(v_rows), slots)

    def copy(self, pairs):
        if not pairs:
            return
        src = torch.tensor([s for s, _ in pairs], dtype=torch.int32, device="cuda")
        dst = torch.tensor([d for _, d in pairs], dtype=torch.int32, device="cuda")
        api.copy_blocks(self.k, src, dst)
        api.copy_blocks(self.v, src, dst)
        self.kc, self.vc = km.copy_blocks(self.kc, pairs), km.copy_blocks(self.vc, pairs)

    def check_bits(self, what):
        assert np.array_equal(synth.bf16_bits(self.k), self.kc), f"{what}: K cache"
        assert np.array_equal(synth.bf16_bits(self.v), self.vc), f"{what}: V cache"


def test_decode_loop_with_allocator_growth_window_recycling_and_fork():
    gen = torch.Generator().manual_seed(71)
    rng = np.random.default_rng(71)
    nb = [48, 28]  # full-attention pool, sliding pool (each with its null block)
    orders = [rng.permutation(n).astype(np.int32) for n in nb]
    lib = api.KVCacheManager([0, WINDOW], nb, BS, MAXB * BS, initial_orders=orders)
    orc = km.KVCacheManager([0, WINDOW], nb, BS, MAXB * BS, initial_orders=orders)
    layers = [Layer(nb[0], gen, 0), Layer(nb[1], gen, WINDOW)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / np.sqrt(D)

    def same_tables(reqs, what):
        for t in range(2):
            got = lib.block_table(t, reqs, MAXB)
            assert np.array_equal(got, orc.block_table(t, reqs, MAXB)), f"{what}: table {t}"
        for r in reqs:
            assert lib.get_block_ids(r) == orc.get_block_ids(r), f"{what}: blocks of {r}"

    def prompt(r, n):
        assert lib.allocate_slots(r, 0, n) and orc.allocate_slots(r, 0, n)
        same_tables([r], f"prompt {r}")
        kr = [_rand_bf16((n, HKV, D), gen) for _ in range(2)]
        vr = [_rand_bf16((n, HKV, D), gen) for _ in range(2)]
        for t, layer in enumerate(layers):
            table = lib.block_table(t, [r], MAXB)
            slots = api.build_slot_mapping(table, [0], [n], BS)
            assert np.array_equal(slots, bp.slot_mapping(table, [0], [n], BS))
            layer.write(slots, kr[t], vr[t], status)

    # Prompts: one just below a block edge, one across two blocks, one token.
    kv_len = {0: 120, 1: 250, 2: 1}
    for r, n in kv_len.items():
        prompt(r, n)
    crossed, recycled = set(), 0
    for step in range(STEPS):
        if step == FORK_AT:  # request 1 forks into 3 and 4 (full blocks shared, the last copied)
            n = kv_len[1]
            got = lib.fork(1, [3, 4], n, True)
            assert got == orc.fork(1, [3, 4], n, True)
            for t, layer in enumerate(layers):
                layer.copy(got[t])
            kv_len[3] = kv_len[4] = n
        if step == SWAP_AT:  # request 2 finishes; request 5 arrives with a prompt
            lib.free(2)
            orc.free(2)
            del kv_len[2]
            prompt(5, 200)
            kv_len[5] = 200
        reqs = sorted(kv_len)
        null_s = lib.null_block(1)
        for r in reqs:
            before = lib.get_block_ids(r)[1]
            ok = lib.allocate_slots(r, kv_len[r], 1)
            assert ok == orc.allocate_slots(r, kv_len[r], 1) and ok, f"step {step}: request {r}"
            after = lib.get_block_ids(r)[1]
            # sliding blocks that left the window went back to the pool as null entries
            recycled += sum(1 for a, b in zip(before, after) if a != null_s and b == null_s)
            if kv_len[r] % BS == 0 and kv_len[r] > 0:
                crossed.add(r)
        assert lib.format_usage() == orc.format_usage()
        same_tables(reqs, f"step {step}")
        starts = [kv_len[r] for r in reqs]
        lens = np.array([kv_len[r] + 1 for r in reqs], dtype=np.int32)
        for t, layer in enumerate(layers):
            table = lib.block_table(t, reqs, MAXB)
            slots = api.build_slot_mapping(table, starts, [1] * len(reqs), BS)
            assert np.array_equal(slots, bp.slot_mapping(table, starts, [1] * len(reqs), BS))
            layer.write(slots, _rand_bf16((len(reqs), HKV, D), gen),
                        _rand_bf16((len(reqs), HKV, D), gen), status)
            q = _rand_bf16((len(reqs), H, D), gen)
            lse = torch.full((len(reqs), H), float("nan"), device="cuda")
            out = api.paged_attention_decode(q.cuda(), layer.k, layer.v,
                                             torch.from_numpy(table).cuda(),
                                             torch.from_numpy(lens).cuda(), scale, layer.window,
                                             lse=lse, dev_status=status)
            torch.cuda.synchronize()
            layer.check_bits(f"step {step} type {t}")
            q64 = ref.bf16_bits_to_f64(synth.bf16_bits(q))
            o_ref, lse_ref = ref.paged_decode(q64, layer.kc, layer.vc, table, lens, BS, scale,
                                              layer.window)
            compare(out, lse, o_ref, lse_ref, list(range(len(reqs))),
                    f"step {step} type {t} requests {reqs}")
        assert int(status.item()) == 0
        for r in reqs:
            kv_len[r] += 1
    # The run did what it is meant to cover.
    assert crossed >= {0, 1, 3, 4, 5}, crossed
    assert recycled > 0  # the sliding pool got blocks back while requests were live
    assert kv_len[0] == 120 + STEPS and kv_len[3] == 250 + FORK_AT + (STEPS - FORK_AT)
    print(f"lifecycle: {STEPS} steps, final kv_len {kv_len}, sliding blocks recycled {recycled}, "
          f"usage {lib.format_usage()}")
