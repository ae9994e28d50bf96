"""GPU parity: absorbed MLA decode (latent 512 + rope 64) vs the fp64 oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import DecodeCase, compare, oracle_mla_all

pytestmark = pytest.mark.gpu

MLA = synth.WORKLOADS["mla"]


def _run(case: DecodeCase, rows, out_dtype=torch.float32, poison_tails=False):
    """GPU write + decode; the oracle's rows `rows` (None: every sequence, run one
    sequence per task in a process pool on the host's cores)."""
    wl = case.wl
    case.gpu_write()
    case.oracle_write()
    if poison_tails:
        torch.cuda.synchronize()
        case.check_write_bit_exact()
        case.poison_tails()
    lse = torch.full((wl.batch, wl.num_heads), float("nan"), device="cuda")
    out = api.mla_paged_decode(case.v["q_nope"], case.v["q_rope"], case.v["cache_nope"],
                               case.v["cache_rope"], case.table, case.seq_lens, wl.scale, lse=lse,
                               out_dtype=out_dtype, dev_status=case.status)
    torch.cuda.synchronize()
    case.check_write_bit_exact()
    if rows is None:
        return (out, lse) + oracle_mla_all(case)
    o_ref, lse_ref = ref.mla_decode(case.v["q_nope"].double().cpu().numpy(),
                                    case.v["q_rope"].double().cpu().numpy(),
                                    case.post["cache_nope"], case.post["cache_rope"], case.table_np,
                                    case.d.seq_lens, wl.block_size, wl.scale, batch_indices=rows)
    return out, lse, o_ref, lse_ref


@pytest.mark.parametrize("H", [128, 16])
def test_mla_small_edge_cases(H):
    lens = [1, 31, 32, 33, 127, 128, 129, 0, 1000, 5000]
    wl = MLA.scaled(batch=len(lens), num_heads=H, seed=31)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens))
    out, lse, o_ref, lse_ref = _run(case, list(range(len(lens))))
    compare(out, lse, o_ref, lse_ref, list(range(len(lens))), f"mla H{H}")
    assert out[7].abs().max().item() == 0.0 and torch.isinf(lse[7]).all()


def test_mla_ignores_nan_in_unwritten_rows():
    lens = [1, 31, 33, 129, 1000, 4095]
    wl = MLA.scaled(batch=len(lens), num_heads=128, seed=33)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens))
    out, lse, o_ref, lse_ref = _run(case, list(range(len(lens))), poison_tails=True)
    compare(out, lse, o_ref, lse_ref, list(range(len(lens))), "mla NaN tails")


def test_mla_bf16_output_long_sequences():
    lens = [8192, 7000, 4096, 3]
    wl = MLA.scaled(batch=4, seed=32)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens))
    out, lse, o_ref, lse_ref = _run(case, [0, 1, 2, 3], out_dtype=torch.bfloat16)
    compare(out, lse, o_ref, lse_ref, [0, 1, 2, 3], "mla bf16")


def test_mla_workload_full_size():
    case = DecodeCase(MLA)
    out, lse, o_ref, lse_ref = _run(case, None)
    rows = list(range(MLA.batch))
    mx, mean = compare(out, lse, o_ref, lse_ref, rows, "mla full")
    print(f"mla full: {len(rows)} of {MLA.batch} sequences, max abs {mx:.2e} mean abs {mean:.2e}")


def test_mla_rope_term_matters_on_gpu():
    # Zero q_nope: the scores come from the rope term alone; the output still
    # averages the nope rows. Dropping the rope term would give the plain mean.
    lens = [300]
    wl = MLA.scaled(batch=1, num_heads=128, seed=33)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens), poison=False)
    case.v["q_nope"].zero_()
    out, lse, o_ref, lse_ref = _run(case, [0])
    compare(out, lse, o_ref, lse_ref, [0], "rope only")
    table = case.table_np
    nope = ref.gather_sequence(case.post["cache_nope"], table[0], 300, 128)[:, 0]
    plain_mean = nope.mean(axis=0)
    assert np.abs(out[0, 0].cpu().numpy() - plain_mean).max() > 1e-2
