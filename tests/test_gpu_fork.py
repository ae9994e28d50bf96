"""GPU parity: block copies of a fork, and decode after a fork, against the oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import kv_manager_ref as km
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import compare

pytestmark = pytest.mark.gpu

BS, HKV, D, H = 128, 8, 128, 32


def _rand_bf16(shape, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def test_copy_blocks_bit_exact():
    gen = torch.Generator().manual_seed(61)
    nb = 300
    cache = _rand_bf16((nb, BS, HKV, D), gen).cuda()
    pre = synth.bf16_bits(cache)
    rng = np.random.default_rng(61)
    perm = rng.permutation(nb)
    src, dst = perm[:40].astype(np.int32), perm[40:80].astype(np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.copy_blocks(cache, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), dev_status=st)
    torch.cuda.synchronize()
    assert np.array_equal(synth.bf16_bits(cache), km.copy_blocks(pre, list(zip(src, dst))))
    assert int(st.item()) == 0


def test_copy_blocks_bad_ids_are_skipped_and_flagged():
    gen = torch.Generator().manual_seed(62)
    nb = 20
    cache = _rand_bf16((nb, BS, 1, 64), gen).cuda()
    pre = synth.bf16_bits(cache)
    src = torch.tensor([3, 25, -1, 4], dtype=torch.int32, device="cuda")
    dst = torch.tensor([7, 8, 9, 20], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.copy_blocks(cache, src, dst, dev_status=st)
    torch.cuda.synchronize()
    assert np.array_equal(synth.bf16_bits(cache), km.copy_blocks(pre, [(3, 7)]))
    assert int(st.item()) & 2  # PKV_DEV_BAD_BLOCK


@pytest.mark.parametrize("prompt_len", [300, 256, 1])
def test_decode_after_fork_matches_oracle(prompt_len):
    """Parent prompt -> fork to two children (shared full blocks, copied last block)
    -> every request appends its own token -> decode. Each child must attend over
    the parent's prompt plus its own token, and the parent must be unaffected."""
    gen = torch.Generator().manual_seed(63 + prompt_len)
    rng = np.random.default_rng(63 + prompt_len)
    nb = 64
    order = rng.permutation(nb).astype(np.int32)
    lib = api.KVCacheManager([0], [nb], BS, 1 << 20, initial_orders=[order])
    orc = km.KVCacheManager([0], [nb], BS, 1 << 20, initial_orders=[order])
    k_cache = _rand_bf16((nb, BS, HKV, D), gen).cuda()
    v_cache = _rand_bf16((nb, BS, HKV, D), gen).cuda()
    kc, vc = synth.bf16_bits(k_cache), synth.bf16_bits(v_cache)
    k_prompt, v_prompt = _rand_bf16((prompt_len, HKV, D), gen), _rand_bf16((prompt_len, HKV, D), gen)
    P, C1, C2 = 10, 11, 12
    reqs = [P, C1, C2]
    maxb = 8

    def slots_for(r, start, n):
        table = lib.block_table(0, [r], maxb)
        assert np.array_equal(table, orc.block_table(0, [r], maxb))
        return api.build_slot_mapping(table, [start], [n], BS)

    def write(r, start, kr, vr):
        nonlocal kc, vc
        s = slots_for(r, start, kr.shape[0])
        api.kv_cache_write(k_cache, v_cache, kr.cuda(), vr.cuda(), torch.from_numpy(s).cuda())
        kc = ref.cache_write(kc, synth.bf16_bits(kr), s)
        vc = ref.cache_write(vc, synth.bf16_bits(vr), s)

    assert lib.allocate_slots(P, 0, prompt_len) and orc.allocate_slots(P, 0, prompt_len)
    write(P, 0, k_prompt, v_prompt)
    pairs = lib.fork(P, [C1, C2], prompt_len, shareable=True)[0]
    assert pairs == orc.fork(P, [C1, C2], prompt_len, True)[0]
    assert len(pairs) == (2 if prompt_len % BS else 0)
    if pairs:
        src = torch.tensor([s for s, _ in pairs], dtype=torch.int32, device="cuda")
        dst = torch.tensor([d for _, d in pairs], dtype=torch.int32, device="cuda")
        api.copy_blocks(k_cache, src, dst)
        api.copy_blocks(v_cache, src, dst)
        kc, vc = km.copy_blocks(kc, pairs), km.copy_blocks(vc, pairs)
    new_k = {r: _rand_bf16((1, HKV, D), gen) for r in reqs}
    new_v = {r: _rand_bf16((1, HKV, D), gen) for r in reqs}
    for r in reqs:
        assert lib.allocate_slots(r, prompt_len, 1) and orc.allocate_slots(r, prompt_len, 1)
        write(r, prompt_len, new_k[r], new_v[r])
    torch.cuda.synchronize()
    assert np.array_equal(synth.bf16_bits(k_cache), kc)
    assert np.array_equal(synth.bf16_bits(v_cache), vc)

    table = lib.block_table(0, reqs, maxb)
    lens = np.full(3, prompt_len + 1, dtype=np.int32)
    q = _rand_bf16((3, H, D), gen)
    scale = 1.0 / np.sqrt(D)
    out = api.paged_attention_decode(q.cuda(), k_cache, v_cache, torch.from_numpy(table).cuda(),
                                     torch.from_numpy(lens).cuda(), scale)
    torch.cuda.synchronize()
    q64 = ref.bf16_bits_to_f64(synth.bf16_bits(q))
    o_ref, lse_ref = ref.paged_decode(q64, kc, vc, table, lens, BS, scale)
    compare(out, None, o_ref, lse_ref, [0, 1, 2], f"decode after fork (prompt {prompt_len})")
    # The fork's meaning, without paging: each request sees the prompt plus its own token.
    for b, r in enumerate(reqs):
        K = ref.bf16_bits_to_f64(np.concatenate([synth.bf16_bits(k_prompt), synth.bf16_bits(new_k[r])]))
        V = ref.bf16_bits_to_f64(np.concatenate([synth.bf16_bits(v_prompt), synth.bf16_bits(new_v[r])]))
        for h in (0, 13, 31):
            o, _, _ = ref.attend(q64[b, h], K[:, h // (H // HKV)], V[:, h // (H // HKV)],
                                 np.ones(prompt_len + 1, dtype=bool), scale)
            assert np.abs(o - o_ref[b, h]).max() < 1e-12
