"""GPU calls on empty batches: no rows to write, no sequences to decode.

A serving step can have no decode requests (all sequences in prefill) or no new
tokens for some layer's cache. Every entry point accepts such a call, launches
nothing that touches memory, returns an empty output of the right shape and leaves
the device status clear; the cache is unchanged.
"""
import pytest
import torch

from paged_kv_cache_77_gb300 import api

pytestmark = pytest.mark.gpu

NB, BS, HKV, D, H = 4, 128, 2, 128, 8


def _bf16(*shape):
    return torch.randn(shape, device="cuda").to(torch.bfloat16)


def _i32(*shape):
    return torch.zeros(shape, dtype=torch.int32, device="cuda")


@pytest.fixture
def status():
    return _i32(1)


def test_empty_writes_leave_the_cache_unchanged(status):
    k, v = _bf16(NB, BS, HKV, D), _bf16(NB, BS, HKV, D)
    k0, v0 = k.clone(), v.clone()
    api.kv_cache_write(k, v, _bf16(0, HKV, D), _bf16(0, HKV, D), _i32(0), dev_status=status)
    kc = torch.zeros((NB, BS, HKV, D), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros((NB, HKV, BS), device="cuda")
    vs = torch.zeros_like(ks)
    api.kv_cache_write_fp8(kc, vc, ks, vs, _bf16(0, HKV, D), _bf16(0, HKV, D), _i32(0),
                           dev_status=status)
    nope, rope = _bf16(NB, BS, 1, 512), _bf16(NB, BS, 1, 64)
    n0, r0 = nope.clone(), rope.clone()
    cs = torch.zeros(0, 64, device="cuda")
    api.mla_rmsnorm_rope_write(nope, rope, _bf16(0, 576), _bf16(512), cs, cs.clone(), _i32(0), 1e-6,
                               dev_status=status)
    api.copy_blocks(k, _i32(0), _i32(0), dev_status=status)
    torch.cuda.synchronize()
    assert torch.equal(k, k0) and torch.equal(v, v0)
    assert torch.equal(nope, n0) and torch.equal(rope, r0)
    assert int(kc.count_nonzero()) == 0 and int(ks.count_nonzero()) == 0
    assert int(status.item()) == 0


def test_empty_decode_batches(status):
    k, v = _bf16(NB, BS, HKV, D), _bf16(NB, BS, HKV, D)
    table, lens = _i32(0, 4), _i32(0)
    out = api.paged_attention_decode(_bf16(0, H, D), k, v, table, lens, 0.1,
                                     lse=torch.empty(0, H, device="cuda"), dev_status=status)
    assert out.shape == (0, H, D)
    out = api.paged_attention_decode(_bf16(0, H, D), k, v, table, lens, 0.1, 64,
                                     out_dtype=torch.bfloat16, dev_status=status)
    assert out.shape == (0, H, D) and out.dtype == torch.bfloat16
    out = api.paged_attention_decode_spec(_bf16(0, 3, H, D), k, v, table, lens, 0.1, dev_status=status)
    assert out.shape == (0, 3, H, D)
    kc = torch.zeros((NB, BS, HKV, D), dtype=torch.uint8, device="cuda")
    ks = torch.ones((NB, HKV, BS), device="cuda")
    out = api.paged_attention_decode_fp8(_bf16(0, H, D), kc, kc.clone(), ks, ks.clone(), table,
                                         lens, 0.1, dev_status=status)
    assert out.shape == (0, H, D)
    nope, rope = _bf16(NB, BS, 1, 512), _bf16(NB, BS, 1, 64)
    out = api.mla_paged_decode(_bf16(0, 16, 512), _bf16(0, 16, 64), nope, rope, table, lens, 0.1,
                               dev_status=status)
    assert out.shape == (0, 16, 512)
    out = api.mla_paged_decode_spec(_bf16(0, 2, 16, 512), _bf16(0, 2, 16, 64), nope, rope, table,
                                    lens, 0.1, dev_status=status)
    assert out.shape == (0, 2, 16, 512)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_prefill_without_new_rows(status):
    k, v = _bf16(NB, BS, HKV, D), _bf16(NB, BS, HKV, D)
    # Two sequences with cached context and no new rows, then no sequences at all.
    for B in (2, 0):
        cu = _i32(B)
        lens = torch.full((B,), 100, dtype=torch.int32, device="cuda")
        table = torch.arange(B * 2, dtype=torch.int32, device="cuda").reshape(B, 2)
        out = api.paged_attention_prefill(_bf16(0, H, D), cu, k, v, table, lens, 0.1,
                                          lse=torch.empty(0, H, device="cuda"), dev_status=status)
        assert out.shape == (0, H, D)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
