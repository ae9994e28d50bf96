"""GPU test of the decode entry point that needs no caller-allocated scratch.

Some callers of this library cannot allocate device memory: a plugin inside a
runtime that owns the device allocator, a serving loop whose HBM is already split
between weights and the KV cache, or code that must avoid the device
synchronisation a cudaMalloc can cause. pkv_paged_attention_decode_static serves
them by keeping its split-KV partials in a fixed array inside the library. This
test calls it through the C ABI twice in a row, on different inputs, and checks
each result against the workspace-taking entry point. It sits in a file that
pytest collects last so that a failure here leaves every other test already run.
"""
import pytest
import torch

import synth
from paged_kv_cache_77_gb300 import api
from paged_kv_cache_77_gb300._lib import PagedKVError
from tests.gpu_cases import MAX_ABS_TOL, MEAN_ABS_TOL, DecodeCase

pytestmark = pytest.mark.gpu


def _check(got, want, lse_got, lse_want):
    err = (got - want).abs()
    assert torch.isfinite(got).all()
    assert err.max().item() <= MAX_ABS_TOL and err.mean().item() <= MEAN_ABS_TOL
    fin = torch.isfinite(lse_want)
    assert torch.equal(torch.isfinite(lse_got), fin)
    assert (lse_got[fin] - lse_want[fin]).abs().max().item() <= 2e-3


def test_static_scratch_decode_matches_workspace_decode_twice():
    # Long sequences so that segments are split across CTAs and the partials (the
    # scratch) are actually written and merged.
    lens = [20000, 15000, 3000, 1, 0, 9000]
    wl = synth.WORKLOADS["gqa_long"].scaled(batch=len(lens), seed=21)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens), poison=True)
    assert api.decode_workspace_size(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim) \
        <= api.STATIC_SCRATCH_BYTES
    q2 = torch.randn_like(case.v["q"], dtype=torch.float32).to(torch.bfloat16)
    for q in (case.v["q"], q2):  # two calls in a row; the second reuses the array
        lse_a = torch.empty((wl.batch, wl.num_heads), device="cuda")
        lse_b = torch.empty_like(lse_a)
        want = api.paged_attention_decode(q, case.v["k_cache"], case.v["v_cache"], case.table,
                                          case.seq_lens, wl.scale, lse=lse_a)
        got = api.paged_attention_decode_static(q, case.v["k_cache"], case.v["v_cache"], case.table,
                                                case.seq_lens, wl.scale, lse=lse_b)
        torch.cuda.synchronize()
        _check(got, want, lse_b, lse_a)


def test_static_scratch_decode_rejects_oversized_problems():
    wl = synth.WORKLOADS["gqa_long"].scaled(batch=4000, seed=22)
    assert api.decode_workspace_size(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim) \
        > api.STATIC_SCRATCH_BYTES
    q = torch.zeros((wl.batch, wl.num_heads, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((2, 128, wl.num_kv_heads, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((wl.batch, 1), dtype=torch.int32, device="cuda")
    lens = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    with pytest.raises(PagedKVError) as e:
        api.paged_attention_decode_static(q, cache, cache, table, lens, wl.scale)
    assert "static" in str(e.value)
