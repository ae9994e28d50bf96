"""GPU parity: absorbed MLA decode of several new rows per sequence (bottom-right
causal) vs the fp64 oracle.

The q_len new latent rows are written through slot_mapping (bit-exact against the
oracle's write), the tails of the last blocks are poisoned with NaN, and every row,
at the small cases and at the full-size workload, is compared with
oracle.mla_spec_decode. Lengths below q_len put rows at negative positions,
which must come back as o = 0, lse = -inf.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from paged_kv_cache_77_gb300._lib import PagedKVError
from tests.gpu_cases import DecodeCase, compare, oracle_mla_all

pytestmark = pytest.mark.gpu

MLA_SPEC = synth.WORKLOADS["mla_spec"]


def _case(Q, H, lens, seed, poison=True):
    wl = MLA_SPEC.scaled(batch=len(lens), num_heads=H, q_lo=Q, q_hi=Q, seed=seed)
    lens = np.asarray(lens)
    return DecodeCase(wl, synth.draw_explicit(wl, lens, num_new=np.minimum(lens, Q)), poison=poison)


def _run(case: DecodeCase, rows, out_dtype=torch.float32, poison_tails=True):
    wl = case.wl
    Q = wl.q_hi
    case.gpu_write()
    case.oracle_write()
    torch.cuda.synchronize()
    case.check_write_bit_exact()
    if poison_tails:
        case.poison_tails()
    lse = torch.full((wl.batch, Q, wl.num_heads), float("nan"), device="cuda")
    out = api.mla_paged_decode_spec(case.v["q_nope"], case.v["q_rope"], case.v["cache_nope"],
                                    case.v["cache_rope"], case.table, case.seq_lens, wl.scale,
                                    lse=lse, out_dtype=out_dtype, dev_status=case.status)
    torch.cuda.synchronize()
    assert int(case.status.item()) == 0
    if rows is None:  # every sequence, one per task in a process pool on the host's cores
        return (out, lse) + oracle_mla_all(case)
    o_ref, lse_ref = ref.mla_spec_decode(case.v["q_nope"].double().cpu().numpy(),
                                         case.v["q_rope"].double().cpu().numpy(),
                                         case.post["cache_nope"], case.post["cache_rope"],
                                         case.table_np, case.d.seq_lens, wl.block_size, wl.scale,
                                         batch_indices=rows)
    return out, lse, o_ref, lse_ref


# Lengths below q_len, and around the 64-token tile and 128-token block edges, where
# the rows of one sequence end in different tiles.
LENS = [0, 1, 2, 3, 4, 5, 63, 64, 65, 66, 67, 127, 128, 129, 130, 131, 1000, 4097]


@pytest.mark.parametrize("Q", [2, 3, 4])
@pytest.mark.parametrize("H", [128, 16])
def test_mla_spec_small_edge_cases(Q, H):
    case = _case(Q, H, LENS, seed=40 + Q)
    rows = list(range(len(LENS)))
    out, lse, o_ref, lse_ref = _run(case, rows)
    compare(out, lse, o_ref, lse_ref, rows, f"mla spec Q{Q} H{H}")
    for b, n in enumerate(LENS):
        for i in range(Q):
            if n - Q + i < 0:
                assert out[b, i].abs().max().item() == 0.0 and torch.isinf(lse[b, i]).all()


def test_mla_spec_q_len_one_equals_decode_entry_bitwise():
    lens = [1, 65, 129, 3000, 8192]
    case = _case(1, 128, lens, seed=45, poison=False)
    case.gpu_write()
    torch.cuda.synchronize()
    wl = case.wl
    q_nope, q_rope = case.v["q_nope"], case.v["q_rope"]  # [B, H, ...] at q_len 1
    a = api.mla_paged_decode_spec(q_nope[:, None].contiguous(), q_rope[:, None].contiguous(),
                                  case.v["cache_nope"], case.v["cache_rope"], case.table,
                                  case.seq_lens, wl.scale)
    b = api.mla_paged_decode(q_nope, q_rope, case.v["cache_nope"], case.v["cache_rope"],
                             case.table, case.seq_lens, wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(a[:, 0], b)


def test_mla_spec_bf16_output_long_sequences():
    lens = [8192, 7001, 4096, 2, 1]
    case = _case(4, 128, lens, seed=46)
    rows = list(range(len(lens)))
    out, lse, o_ref, lse_ref = _run(case, rows, out_dtype=torch.bfloat16)
    compare(out, lse, o_ref, lse_ref, rows, "mla spec bf16")


def test_mla_spec_rejects_unsupported_q_len():
    case = _case(2, 16, [10, 20], seed=47, poison=False)
    q5 = torch.zeros((2, 5, 16, 512), dtype=torch.bfloat16, device="cuda")
    r5 = torch.zeros((2, 5, 16, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(PagedKVError):
        api.mla_paged_decode_spec(q5, r5, case.v["cache_nope"], case.v["cache_rope"], case.table,
                                  case.seq_lens, case.wl.scale)


def test_mla_spec_workload_full_size():
    case = DecodeCase(MLA_SPEC)
    out, lse, o_ref, lse_ref = _run(case, None)
    rows = list(range(MLA_SPEC.batch))
    mx, mean = compare(out, lse, o_ref, lse_ref, rows, "mla spec full")
    print(f"mla spec full: {len(rows)} of {MLA_SPEC.batch} sequences x {MLA_SPEC.q_hi} rows, "
          f"max abs {mx:.2e} mean abs {mean:.2e}")


@pytest.mark.parametrize("H,Q", [(1, 4), (40, 2), (40, 3)])
def test_mla_spec_head_counts_below_the_tile(H, Q):
    # The 128-row Q box reaches past the last row of q when H < 128; those rows must
    # neither be read as data nor written.
    lens = [1, 4, 64, 65, 200, 777, 3000]
    case = _case(Q, H, lens, seed=50 + H + Q)
    rows = list(range(len(lens)))
    out, lse, o_ref, lse_ref = _run(case, rows)
    compare(out, lse, o_ref, lse_ref, rows, f"mla spec H{H} Q{Q}")


def test_mla_spec_many_short_rows_split_across_pairs():
    # 64 sequences of 0..300 positions at q_len 4: 256 rows, most of them cut by pair
    # range boundaries (a few tiles per pair), empty rows in between.
    rng = np.random.default_rng(57)
    lens = rng.integers(0, 300, size=64)
    lens[::9] = 0
    case = _case(4, 128, lens.tolist(), seed=57)
    rows = list(range(len(lens)))
    out, lse, o_ref, lse_ref = _run(case, rows)
    compare(out, lse, o_ref, lse_ref, rows, "mla spec many short rows")
