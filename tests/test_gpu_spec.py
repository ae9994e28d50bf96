"""GPU parity: speculative (multi-token) decode vs the fp64 oracle.

q_len new rows per sequence are written through slot_mapping (bit-exact against
the oracle's write), the tails of the last blocks are poisoned with NaN, and the
tensor-core kernel's output is compared with oracle.paged_spec_decode on every
row, at the small cases and at the full-size workload."""
import numpy as np
import pytest
import torch

import synth
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import DecodeCase, compare, oracle_decode_all

pytestmark = pytest.mark.gpu

SPEC = synth.WORKLOADS["spec_decode"]


def _run(case: DecodeCase, rows, out_dtype=torch.float32, poison=True):
    wl = case.wl
    case.gpu_write()
    case.oracle_write()
    case.check_write_bit_exact()
    if poison:
        case.poison_tails()
    Q = wl.q_hi
    lse = torch.full((wl.batch, Q, wl.num_heads), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.paged_attention_decode_spec(case.v["q"], case.v["k_cache"], case.v["v_cache"],
                                          case.table, case.seq_lens, wl.scale, wl.window, lse=lse,
                                          out_dtype=out_dtype, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    q64 = case.v["q"].double().cpu().numpy()
    o_ref, lse_ref = ref.paged_spec_decode(q64, case.post["k_cache"], case.post["v_cache"],
                                           case.table_np, case.d.seq_lens, wl.block_size, wl.scale,
                                           wl.window, batch_indices=rows)
    return out, lse, o_ref, lse_ref


def _lens_case(H, Hkv, Q, window, lens, seed):
    wl = SPEC.scaled(batch=len(lens), num_heads=H, num_kv_heads=Hkv, q_lo=Q, q_hi=Q,
                     window=window, seed=seed)
    lens = np.asarray(lens)
    d = synth.draw_explicit(wl, lens, num_new=np.minimum(lens, Q))
    return DecodeCase(wl, d)


# Every column layout of the kernel: rows per kv head 4, 6, 8, 16 (N = 16) and
# 24, 32 (N = 32, two softmax warp groups), from 1, 2, 4, 8 and 16 heads per group.
SHAPES = [(4, 4, 4), (8, 4, 3), (16, 4, 2), (16, 4, 4), (32, 4, 2), (32, 4, 3), (32, 4, 4),
          (32, 2, 2)]


@pytest.mark.parametrize("H,Hkv,Q", SHAPES)
@pytest.mark.parametrize("window", [0, 200])
def test_spec_decode_small_edge_cases(H, Hkv, Q, window):
    # Lengths below q_len (rows at negative positions), at and around block edges,
    # an empty sequence, and long enough to split over several CTAs.
    lens = [1, 3, 4, 127, 128, 129, 130, 700, 0, 2000, 255, 5]
    case = _lens_case(H, Hkv, Q, window, lens, seed=31 + Q)
    rows = list(range(len(lens)))
    out, lse, o_ref, lse_ref = _run(case, rows)
    compare(out, lse, o_ref, lse_ref, rows, f"spec H{H}/Hkv{Hkv}/Q{Q}/W{window}")
    assert out[8].abs().max().item() == 0.0 and torch.isinf(lse[8]).all()  # empty sequence


def test_spec_decode_bf16_output_and_many_splits():
    lens = [5000, 4, 4096, 12000]
    case = _lens_case(64, 8, 4, 0, lens, seed=41)
    out, lse, o_ref, lse_ref = _run(case, [0, 1, 2, 3], out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16
    compare(out, lse, o_ref, lse_ref, [0, 1, 2, 3], "spec bf16 out")


def test_spec_decode_q_len_one_is_the_decode_kernel():
    lens = [1, 129, 700, 3000]
    case = _lens_case(64, 8, 1, 0, lens, seed=42)
    case.gpu_write()
    wl = case.wl
    q = case.v["q"]  # [B, 1, H, d]
    a = api.paged_attention_decode_spec(q, case.v["k_cache"], case.v["v_cache"], case.table,
                                        case.seq_lens, wl.scale)
    api.set_decode_kernel(api.KERNEL_TENSOR_CORE)
    try:
        b = api.paged_attention_decode(q[:, 0].contiguous(), case.v["k_cache"], case.v["v_cache"],
                                       case.table, case.seq_lens, wl.scale)
    finally:
        api.set_decode_kernel(api.KERNEL_AUTO)
    torch.cuda.synchronize()
    assert torch.equal(a[:, 0], b)


@pytest.mark.parametrize("window", [0, 4096])
def test_spec_decode_full_size(window):
    """The bench's workload (64 sequences up to 32768 tokens, 64 heads over 8 kv
    heads, 4 new rows each): every row compared with the oracle, run one sequence
    per task in a process pool on the host's cores."""
    wl = SPEC.scaled(window=window)
    case = DecodeCase(wl, synth.draw(wl))
    case.gpu_write()
    case.oracle_write()
    case.check_write_bit_exact()
    case.poison_tails()
    lse = torch.full((wl.batch, wl.q_hi, wl.num_heads), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.paged_attention_decode_spec(case.v["q"], case.v["k_cache"], case.v["v_cache"],
                                          case.table, case.seq_lens, wl.scale, wl.window, lse=lse,
                                          dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, lse_ref = oracle_decode_all(case)
    rows = list(range(wl.batch))
    mx, mean = compare(out, lse, o_ref, lse_ref, rows, f"spec full W{window}")
    print(f"spec_decode W{window}: {wl.batch} of {wl.batch} sequences x {wl.q_hi} rows, "
          f"max abs {mx:.2e} mean abs {mean:.2e}")
