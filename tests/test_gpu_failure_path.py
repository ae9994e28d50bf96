"""Failure detection on the GPU without a fault: every mbarrier wait in the attention
kernels is bounded, and one that runs out sets PKV_DEV_TIMEOUT in the caller's status
word instead of hanging. The self-test kernel waits with the same routines on a
barrier that nothing completes; the test checks the status bit, that the wait gave up
after about its limit rather than at once or never, and that the context is still
usable: a decode call afterwards matches the oracle."""
import time

import numpy as np
import pytest
import torch

import synth
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import DecodeCase, compare

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    st.fill_(1)  # other bits are kept
    torch.cuda.synchronize()
    t = time.perf_counter()
    api.selftest_bounded_wait(st)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t
    assert int(st.item()) == 1 | api.DEV_TIMEOUT
    # The limit is 2e9 clock cycles per wait (about a second at 2 GHz; the two waits
    # run side by side).
    assert 0.2 < elapsed < 30.0, elapsed


def test_context_usable_after_a_timeout():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.selftest_bounded_wait(st)
    torch.cuda.synchronize()
    assert int(st.item()) & api.DEV_TIMEOUT
    lens = [1, 300, 2000]
    wl = synth.WORKLOADS["gqa_long"].scaled(batch=3, num_heads=16, num_kv_heads=2, seed=81)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens))
    case.gpu_write()
    case.oracle_write()
    lse = torch.full((wl.batch, wl.num_heads), float("nan"), device="cuda")
    out = api.paged_attention_decode(case.v["q"], case.v["k_cache"], case.v["v_cache"], case.table,
                                     case.seq_lens, wl.scale, lse=lse, dev_status=case.status)
    torch.cuda.synchronize()
    case.check_write_bit_exact()
    o_ref, lse_ref = ref.paged_decode(case.v["q"].double().cpu().numpy(), case.post["k_cache"],
                                      case.post["v_cache"], case.table_np, case.d.seq_lens,
                                      wl.block_size, wl.scale)
    compare(out, lse, o_ref, lse_ref, list(range(3)), "decode after a timeout")


def test_null_status_is_rejected():
    with pytest.raises(ValueError):
        api.selftest_bounded_wait(None)
