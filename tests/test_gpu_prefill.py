"""GPU parity: causal paged prefill (TND queries, bottom-right mask) vs the fp64 oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import PREFILL_LSE_TOL, DecodeCase, compare, oracle_prefill_all

pytestmark = pytest.mark.gpu

MIX = synth.WORKLOADS["mixed_prefill"]


def _case(wl, prior, qlen, poison=True):
    prior, qlen = np.asarray(prior), np.asarray(qlen)
    d = synth.draw_explicit(wl, prior + qlen, num_new=qlen)
    return DecodeCase(wl, d, poison=poison)


def _run(case: DecodeCase, rows, causal=True, out_dtype=torch.float32, poison_tails=False):
    wl = case.wl
    case.gpu_write()
    case.oracle_write()
    if poison_tails:
        torch.cuda.synchronize()
        case.check_write_bit_exact()
        case.poison_tails()
    cu = torch.from_numpy(np.cumsum(case.d.num_new).astype(np.int32)).cuda()
    T = int(case.d.num_new.sum())
    lse = torch.full((T, wl.num_heads), float("nan"), device="cuda")
    out = api.paged_attention_prefill(case.v["q"], cu, case.v["k_cache"], case.v["v_cache"],
                                      case.table, case.seq_lens, wl.scale, causal=causal, lse=lse,
                                      out_dtype=out_dtype, dev_status=case.status)
    torch.cuda.synchronize()
    case.check_write_bit_exact()
    if rows is None:  # every row, in runs of rows per task in a process pool on the host's cores
        return (out, lse) + oracle_prefill_all(case, causal=causal)
    o_ref, lse_ref = ref.paged_prefill(case.v["q"].double().cpu().numpy(), np.cumsum(case.d.num_new),
                                       case.post["k_cache"], case.post["v_cache"], case.table_np,
                                       case.d.seq_lens, wl.block_size, wl.scale, causal=causal,
                                       rows=rows)
    return out, lse, o_ref, lse_ref


@pytest.mark.parametrize("H,Hkv", [(32, 8), (16, 16), (32, 2), (16, 8)])
def test_prefill_small_edge_cases(H, Hkv):
    prior = [0, 5, 0, 200, 1000, 127, 300, 64]
    qlen = [1, 3, 130, 33, 1, 129, 0, 257]
    wl = MIX.scaled(batch=len(prior), num_heads=H, num_kv_heads=Hkv, seed=41)
    case = _case(wl, prior, qlen)
    T = sum(qlen)
    out, lse, o_ref, lse_ref = _run(case, None)
    compare(out, lse, o_ref, lse_ref, list(range(T)), f"prefill H{H}/Hkv{Hkv}",
            lse_tol=PREFILL_LSE_TOL)


def test_prefill_non_causal_differs_and_matches_oracle():
    prior, qlen = [10, 300], [40, 100]
    wl = MIX.scaled(batch=2, seed=42)
    case = _case(wl, prior, qlen)
    out, lse, o_ref, lse_ref = _run(case, None, causal=False)
    compare(out, lse, o_ref, lse_ref, list(range(140)), "non-causal", lse_tol=PREFILL_LSE_TOL)
    # The causal oracle differs on early rows (the pages' error table: prefill
    # without the causal mode gives wrong output).
    o_c, _ = ref.paged_prefill(case.v["q"].double().cpu().numpy(), np.cumsum(qlen),
                               case.post["k_cache"], case.post["v_cache"], case.table_np,
                               case.d.seq_lens, 128, wl.scale, causal=True, rows=[0])
    assert np.abs(o_c[0] - out[0].cpu().numpy()).max() > 1e-2


def test_prefill_ignores_nan_in_unwritten_rows():
    prior, qlen = [0, 5, 200, 1000, 127], [3, 130, 33, 300, 1]
    wl = MIX.scaled(batch=len(prior), num_heads=32, num_kv_heads=8, seed=46)
    T = sum(qlen)
    for causal in (True, False):
        case = _case(wl, prior, qlen)
        out, lse, o_ref, lse_ref = _run(case, None, causal=causal, poison_tails=True)
        compare(out, lse, o_ref, lse_ref, list(range(T)), f"prefill NaN tails causal={causal}",
                lse_tol=PREFILL_LSE_TOL)


def test_prefill_bf16_output():
    prior, qlen = [4000, 0, 77], [600, 300, 1]
    wl = MIX.scaled(batch=3, seed=43)
    case = _case(wl, prior, qlen)
    out, lse, o_ref, lse_ref = _run(case, None, out_dtype=torch.bfloat16)
    compare(out, lse, o_ref, lse_ref, list(range(901)), "prefill bf16", lse_tol=PREFILL_LSE_TOL)


def test_prefill_workload_full_size():
    case = DecodeCase(MIX)
    T = int(case.d.num_new.sum())
    out, lse, o_ref, lse_ref = _run(case, None)
    rows = list(range(T))
    mx, mean = compare(out, lse, o_ref, lse_ref, rows, "mixed_prefill full", lse_tol=PREFILL_LSE_TOL)
    print(f"mixed_prefill: {len(rows)} of {T} query rows, max abs {mx:.2e} mean abs {mean:.2e}")


def test_prefill_rows_equal_decode_steps_on_gpu():
    # "手写40行": one-shot prefill equals token-by-token decode. Row r of a sequence
    # with prior c equals a decode over the first c + r + 1 keys.
    prior, qlen = [50], [300]
    wl = MIX.scaled(batch=1, num_heads=32, num_kv_heads=8, seed=45)
    case = _case(wl, prior, qlen, poison=False)
    out, _, _, _ = _run(case, [0])
    for r in (0, 77, 128, 299):
        lens = torch.tensor([prior[0] + r + 1], dtype=torch.int32, device="cuda")
        dec = api.paged_attention_decode(case.v["q"][r:r + 1].contiguous(), case.v["k_cache"],
                                         case.v["v_cache"], case.table, lens, wl.scale)
        torch.cuda.synchronize()
        assert (dec[0] - out[r]).abs().max().item() < 5e-3
