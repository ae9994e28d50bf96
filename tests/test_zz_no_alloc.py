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


def _reference(case, q, window, out_dtype):
    """The workspace-taking entry point on a NaN-filled workspace: any partial the
    merge read without the attention kernel having written it would show."""
    wl = case.wl
    need = api.decode_workspace_size(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim)
    ws = torch.full((need // 4 + 64,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.empty((wl.batch, wl.num_heads), device="cuda")
    out = api.paged_attention_decode(q, case.v["k_cache"], case.v["v_cache"], case.table,
                                     case.seq_lens, wl.scale, window, lse=lse, out_dtype=out_dtype,
                                     workspace=ws)
    return out, lse


def _static(case, q, window, out_dtype):
    wl = case.wl
    lse = torch.empty((wl.batch, wl.num_heads), device="cuda")
    out = api.paged_attention_decode_static(q, case.v["k_cache"], case.v["v_cache"], case.table,
                                            case.seq_lens, wl.scale, window, lse=lse,
                                            out_dtype=out_dtype)
    return out, lse


def test_static_scratch_decode_matches_workspace_decode_twice():
    # Two calls in a row with different batches, lengths (so different cut points of
    # the split-KV pieces and a different set of scratch slots), window and output
    # type; long sequences so that segments are split across CTAs and the partials in
    # the array are written and merged. Each call is checked against the
    # workspace-taking entry point.
    first = DecodeCase(synth.WORKLOADS["gqa_long"].scaled(batch=6, seed=21),
                       synth.draw_explicit(synth.WORKLOADS["gqa_long"].scaled(batch=6, seed=21),
                                           [20000, 15000, 3000, 1, 0, 9000]), poison=True)
    wl2 = synth.WORKLOADS["gqa_long"].scaled(batch=3, num_heads=32, seed=23)
    second = DecodeCase(wl2, synth.draw_explicit(wl2, [7777, 30001, 129]), poison=True)
    runs = ((first, 0, torch.float32), (second, 4096, torch.bfloat16))
    for case, window, out_dtype in runs:
        wl = case.wl
        assert api.decode_workspace_size(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim) \
            <= api.STATIC_SCRATCH_BYTES
        q = case.v["q"]
        got, lse_got = _static(case, q, window, out_dtype)
        want, lse_want = _reference(case, q, window, out_dtype)
        torch.cuda.synchronize()
        assert got.dtype == out_dtype
        _check(got.float(), want.float(), lse_got, lse_want)


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
