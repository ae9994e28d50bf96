"""The process pool that runs the oracle over the parts of a batch (full-size GPU
parity uses it) gives exactly what one direct oracle call on the whole batch gives.

CPU only: small seeded instances, the pool with two spawned workers."""
from types import SimpleNamespace

import numpy as np
import pytest

import synth
from oracle import block_pool_ref as bp
from oracle import fp8_ref as f8
from oracle import paged_ref as ref
from tests import gpu_cases as gc


def _cpu_case(wl, lens, num_new=None):
    d = synth.draw_explicit(wl, lens, num_new)
    v = synth.values(wl, d, "cpu", poison_null=True)  # as on the GPU: the null block is NaN
    win = wl.window + wl.q_hi - 1 if wl.kind == "spec_decode" and wl.window > 0 else wl.window
    table = bp.prepare_block_tables(bp.BlockPool(d.num_blocks, d.pool_order), d.seq_lens,
                                    wl.block_size, win, d.max_blocks_per_seq)
    slots = bp.slot_mapping(table, d.start_pos, d.num_new, wl.block_size)
    if wl.kind == "mla_decode":
        post = {"cache_nope": ref.cache_write(synth.bf16_bits(v["cache_nope"]),
                                              synth.bf16_bits(v["nope_new"]), slots),
                "cache_rope": ref.cache_write(synth.bf16_bits(v["cache_rope"]),
                                              synth.bf16_bits(v["rope_new"]), slots)}
        pre = None
    else:
        pre = {"k_cache": synth.bf16_bits(v["k_cache"]), "v_cache": synth.bf16_bits(v["v_cache"])}
        post = {"k_cache": ref.cache_write(pre["k_cache"], synth.bf16_bits(v["k_new"]), slots),
                "v_cache": ref.cache_write(pre["v_cache"], synth.bf16_bits(v["v_new"]), slots)}
    return SimpleNamespace(wl=wl, d=d, v=v, table_np=table, slots_np=slots, pre=pre, post=post)


@pytest.fixture(autouse=True)
def two_workers(monkeypatch):
    import oracle.pool

    monkeypatch.setattr(oracle.pool, "default_workers", lambda: 2)


def _same(a, b):
    assert a.shape == b.shape
    assert np.array_equal(np.isnan(a), np.isnan(b))
    assert np.array_equal(np.nan_to_num(a, nan=7.0), np.nan_to_num(b, nan=7.0))


@pytest.mark.parametrize("window", [0, 200])
def test_pool_decode_equals_direct_call(window):
    wl = synth.WORKLOADS["gqa_long"].scaled(batch=4, num_heads=8, num_kv_heads=2, window=window,
                                            seed=61)
    c = _cpu_case(wl, [300, 1, 129, 0])
    o, lse = gc.oracle_decode_all(c)
    o_d, lse_d = ref.paged_decode(c.v["q"].double().numpy(), c.post["k_cache"], c.post["v_cache"],
                                  c.table_np, c.d.seq_lens, 128, wl.scale, window)
    _same(o, o_d)
    _same(lse, lse_d)


def test_pool_spec_decode_equals_direct_call():
    wl = synth.WORKLOADS["spec_decode"].scaled(batch=3, num_heads=8, num_kv_heads=2, seed=62)
    c = _cpu_case(wl, [300, 2, 140], num_new=[wl.q_hi] * 3)
    o, lse = gc.oracle_decode_all(c)
    o_d, lse_d = ref.paged_spec_decode(c.v["q"].double().numpy(), c.post["k_cache"],
                                       c.post["v_cache"], c.table_np, c.d.seq_lens, 128, wl.scale)
    _same(o, o_d)
    _same(lse, lse_d)


@pytest.mark.parametrize("name", ["mla", "mla_spec"])
def test_pool_mla_equals_direct_call(name):
    wl = synth.WORKLOADS[name].scaled(batch=3, num_heads=4, seed=63)
    c = _cpu_case(wl, [70, 1, 200], num_new=[wl.q_hi] * 3)
    o, lse = gc.oracle_mla_all(c)
    fn = ref.mla_spec_decode if name == "mla_spec" else ref.mla_decode
    o_d, lse_d = fn(c.v["q_nope"].double().numpy(), c.v["q_rope"].double().numpy(),
                    c.post["cache_nope"], c.post["cache_rope"], c.table_np, c.d.seq_lens, 128,
                    wl.scale)
    _same(o, o_d)
    _same(lse, lse_d)


@pytest.mark.parametrize("causal", [True, False])
def test_pool_prefill_parts_equal_direct_call(causal):
    # Parts of 5 rows cut every sequence with more than 5 new rows: row r0 + i of a part
    # with c + r0 prior keys must see what row r0 + i of the whole sequence sees.
    wl = synth.WORKLOADS["mixed_prefill"].scaled(batch=4, num_heads=4, num_kv_heads=2, seed=64)
    prior, qlen = np.array([0, 130, 7, 3]), np.array([13, 1, 6, 0])
    c = _cpu_case(wl, prior + qlen, num_new=qlen)
    o, lse = gc.oracle_prefill_all(c, causal=causal, rows_per_part=5)
    o_d, lse_d = ref.paged_prefill(c.v["q"].double().numpy(), np.cumsum(qlen), c.post["k_cache"],
                                   c.post["v_cache"], c.table_np, c.d.seq_lens, 128, wl.scale,
                                   causal=causal)
    # A part gathers fewer keys than its sequence has, and numpy's pairwise sums depend
    # on the array length: equal up to fp64 rounding, not bit for bit.
    assert o.shape == o_d.shape and lse.shape == lse_d.shape
    np.testing.assert_allclose(o, o_d, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_d, rtol=0, atol=1e-12)


@pytest.mark.parametrize("window", [0, 200])
def test_pool_fp8_sequence_equals_whole_cache_oracle(window):
    # The per-sequence FP8 worker (compact cache, remapped table) gives what the oracle
    # gives on the whole quantised cache, and counts every planted code mismatch.
    wl = synth.WORKLOADS["gqa_long"].scaled(batch=3, num_heads=8, num_kv_heads=2, window=window,
                                            seed=65)
    c = _cpu_case(wl, [700, 1, 300])
    codes = {}
    for n, pre, new in (("k", c.pre["k_cache"], c.v["k_new"]), ("v", c.pre["v_cache"], c.v["v_new"])):
        # every block but the NaN null block quantised; the null block holds zeros
        lq, ls = f8.quantize_rows(pre[1:])
        q8 = np.zeros(pre.shape, dtype=np.uint8)
        s8 = np.zeros((pre.shape[0], pre.shape[2], pre.shape[1]), dtype=np.float32)
        q8[1:], s8[1:] = lq, ls.transpose(0, 2, 1)
        q8, s8 = f8.cache_write_fp8(q8, s8, synth.bf16_bits(new), c.slots_np)
        codes[n + "c"], codes[n + "s"] = q8, s8
    o, lse, bad = gc.oracle_fp8_all(c, codes)
    assert bad == 0
    o_d, lse_d = ref.paged_decode(c.v["q"].double().numpy(),
                                  f8.dequantize_cache(codes["kc"], codes["ks"]),
                                  f8.dequantize_cache(codes["vc"], codes["vs"]), c.table_np,
                                  c.d.seq_lens, 128, wl.scale, window)
    np.testing.assert_allclose(o, o_d, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_d, rtol=0, atol=1e-12)
    planted = dict(codes)
    planted["kc"] = codes["kc"].copy()
    live = int(c.table_np[0, (700 - 1) // 128])  # the last block is live at any window
    planted["kc"][live, 3, 1, 5] ^= 1
    assert gc.oracle_fp8_all(c, planted)[2] == 1
