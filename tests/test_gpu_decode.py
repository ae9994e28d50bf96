"""GPU parity: slot_mapping write (bit-exact) and paged decode attention vs the oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import DecodeCase, compare, oracle_decode_all

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["gqa_long"]
KERNELS = {"cuda_core": api.KERNEL_CUDA_CORE, "tensor_core": api.KERNEL_TENSOR_CORE}


@pytest.fixture(params=list(KERNELS))
def kernel(request):
    api.set_decode_kernel(KERNELS[request.param])
    yield request.param
    api.set_decode_kernel(api.KERNEL_AUTO)


def _run_decode(case: DecodeCase, rows, out_dtype=torch.float32):
    wl = case.wl
    case.gpu_write()
    case.oracle_write()
    B = wl.batch
    lse = torch.full((B, wl.num_heads), float("nan"), device="cuda")
    out = api.paged_attention_decode(case.v["q"], case.v["k_cache"], case.v["v_cache"], case.table,
                                     case.seq_lens, wl.scale, wl.window, lse=lse,
                                     out_dtype=out_dtype, dev_status=case.status)
    torch.cuda.synchronize()
    case.check_write_bit_exact()
    q64 = case.v["q"].double().cpu().numpy()
    o_ref, lse_ref = ref.paged_decode(q64, case.post["k_cache"], case.post["v_cache"], case.table_np,
                                      case.d.seq_lens, wl.block_size, wl.scale, wl.window,
                                      batch_indices=rows)
    return out, lse, o_ref, lse_ref


@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 4), (16, 4), (16, 2), (32, 2)])
@pytest.mark.parametrize("window", [0, 200])
def test_decode_small_edge_cases(H, Hkv, window, kernel):
    lens = [1, 127, 128, 129, 700, 0, 2000, 255]
    wl = BASE.scaled(batch=len(lens), num_heads=H, num_kv_heads=Hkv, window=window, seed=7)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens))
    out, lse, o_ref, lse_ref = _run_decode(case, list(range(len(lens))))
    compare(out, lse, o_ref, lse_ref, list(range(len(lens))), f"{kernel} H{H}/Hkv{Hkv}/W{window}")
    assert out[5].abs().max().item() == 0.0 and torch.isinf(lse[5]).all()  # empty sequence


def test_decode_ignores_nan_in_unwritten_rows(kernel):
    # Rows past each sequence's end in its last block are NaN: a masked weight of 0
    # times NaN must not reach the output.
    lens = [1, 129, 700, 3000, 255, 4097]
    wl = BASE.scaled(batch=len(lens), num_heads=32, num_kv_heads=8, window=0, seed=9)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens))
    case.gpu_write()
    case.oracle_write()
    case.check_write_bit_exact()
    case.poison_tails()
    for window in (0, 200):
        lse = torch.full((wl.batch, wl.num_heads), float("nan"), device="cuda")
        out = api.paged_attention_decode(case.v["q"], case.v["k_cache"], case.v["v_cache"], case.table,
                                         case.seq_lens, wl.scale, window, lse=lse)
        torch.cuda.synchronize()
        q64 = case.v["q"].double().cpu().numpy()
        o_ref, lse_ref = ref.paged_decode(q64, case.post["k_cache"], case.post["v_cache"], case.table_np,
                                          case.d.seq_lens, wl.block_size, wl.scale, window)
        compare(out, lse, o_ref, lse_ref, list(range(len(lens))), f"{kernel} NaN tails W{window}")


def test_decode_bf16_output_and_many_splits(kernel):
    lens = [5000, 3, 4096, 12000]
    wl = BASE.scaled(batch=4, num_heads=64, num_kv_heads=8, seed=8)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens))
    out, lse, o_ref, lse_ref = _run_decode(case, [0, 1, 2, 3], out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16
    compare(out, lse, o_ref, lse_ref, [0, 1, 2, 3], "bf16 out")


_FULL_ORACLE = {}  # workload name -> (o, lse): the inputs are seeded, so both kernels share it


@pytest.mark.parametrize("name", ["mha_tiny", "gqa_long", "swa"])
def test_decode_workloads_full_size(name, kernel):
    # Every sequence and head of the workload is compared with the oracle, which runs
    # one sequence per task in a process pool on the host's cores.
    wl = synth.WORKLOADS[name]
    case = DecodeCase(wl)
    case.gpu_write()
    case.oracle_write()
    lse = torch.full((wl.batch, wl.num_heads), float("nan"), device="cuda")
    out = api.paged_attention_decode(case.v["q"], case.v["k_cache"], case.v["v_cache"], case.table,
                                     case.seq_lens, wl.scale, wl.window, lse=lse,
                                     dev_status=case.status)
    torch.cuda.synchronize()
    case.check_write_bit_exact()
    if name not in _FULL_ORACLE:
        _FULL_ORACLE[name] = oracle_decode_all(case)
    o_ref, lse_ref = _FULL_ORACLE[name]
    rows = list(range(wl.batch))
    mx, mean = compare(out, lse, o_ref, lse_ref, rows, f"{kernel} {name}")
    print(f"{kernel} {name}: {len(rows)} of {wl.batch} sequences, max abs {mx:.2e} "
          f"mean abs {mean:.2e}")


def test_worked_slot_marker_row():
    # batch 1, pos 300 on the 2 x 16 arange layout lands in block 18, offset 44 (slot 2348).
    cache = torch.zeros((32, 128, 1, 8), dtype=torch.bfloat16, device="cuda")
    row = torch.arange(1, 9, dtype=torch.float32, device="cuda").to(torch.bfloat16).view(1, 1, 8)
    table = api.build_block_table_arange(2, 16)
    slots = torch.from_numpy(api.build_slot_mapping(table, [0, 300], [0, 1], 128)).cuda()
    assert slots.tolist() == [2348]
    api.kv_cache_write(cache, None, row, None, slots)
    torch.cuda.synchronize()
    assert torch.equal(cache[18, 44, 0], row[0, 0])
    assert cache.float().abs().sum().item() == row.float().sum().item()


def test_paged_equals_contiguous_bitwise(kernel):
    # Same logical KV under the arange table and under a shuffled table: the
    # tile plan depends only on the lengths, so the outputs are bit-identical.
    lens = np.array([900, 130, 4000], dtype=np.int32)
    wl = BASE.scaled(batch=3, num_heads=16, num_kv_heads=2, seed=9)
    d = synth.draw_explicit(wl, lens)
    v = synth.values(wl, d, "cuda")
    nblk = [-(-int(n) // 128) for n in lens]
    per = max(nblk)
    arange_tab = np.zeros((3, per), dtype=np.int32)
    shuf_tab = np.zeros((3, per), dtype=np.int32)
    perm = np.random.default_rng(3).permutation(3 * per)
    k_lin = torch.zeros((3 * per, 128, 2, 128), dtype=torch.bfloat16, device="cuda")
    k_shf, v_lin, v_shf = k_lin.clone(), k_lin.clone(), k_lin.clone()
    for b in range(3):
        for j in range(nblk[b]):
            arange_tab[b, j] = b * per + j
            shuf_tab[b, j] = perm[b * per + j]
            src = v["k_cache"][(b * per + j) % d.num_blocks]
            srcv = v["v_cache"][(b * per + j) % d.num_blocks]
            k_lin[b * per + j] = src
            v_lin[b * per + j] = srcv
            k_shf[perm[b * per + j]] = src
            v_shf[perm[b * per + j]] = srcv
    sl = torch.from_numpy(lens).cuda()
    o1 = api.paged_attention_decode(v["q"], k_lin, v_lin, torch.from_numpy(arange_tab).cuda(), sl,
                                    wl.scale)
    o2 = api.paged_attention_decode(v["q"], k_shf, v_shf, torch.from_numpy(shuf_tab).cuda(), sl,
                                    wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_constant_values_give_constant_output(kernel):
    lens = [1, 333, 5000]
    wl = BASE.scaled(batch=3, num_heads=16, num_kv_heads=2, seed=10)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens), poison=False)
    case.v["v_cache"].fill_(1.0)
    out = api.paged_attention_decode(case.v["q"], case.v["k_cache"], case.v["v_cache"], case.table,
                                     case.seq_lens, wl.scale)
    torch.cuda.synchronize()
    assert (out - 1.0).abs().max().item() < 1e-5


def test_bad_block_and_bad_slot_are_reported_not_read(kernel):
    lens = [300]
    wl = BASE.scaled(batch=1, num_heads=8, num_kv_heads=8, seed=11)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens), poison=False)
    bad = case.table.clone()
    bad[0, 1] = case.d.num_blocks + 5  # out of range: skipped and flagged
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.paged_attention_decode(case.v["q"], case.v["k_cache"], case.v["v_cache"], bad,
                               case.seq_lens, wl.scale, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 2
    st.zero_()
    slots = torch.tensor([case.d.num_blocks * 128 + 3], dtype=torch.int32, device="cuda")
    api.kv_cache_write(case.v["k_cache"], case.v["v_cache"], case.v["k_new"], case.v["v_new"], slots,
                       dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 1


def test_cuda_core_and_tensor_core_kernels_agree():
    lens = [77, 4000, 129, 9000, 1]
    wl = BASE.scaled(batch=5, seed=12)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens), poison=True)
    outs = []
    for k in (api.KERNEL_CUDA_CORE, api.KERNEL_TENSOR_CORE):
        api.set_decode_kernel(k)
        outs.append(api.paged_attention_decode(case.v["q"], case.v["k_cache"], case.v["v_cache"],
                                               case.table, case.seq_lens, wl.scale))
    api.set_decode_kernel(api.KERNEL_AUTO)
    torch.cuda.synchronize()
    # Different accumulation orders (and bf16 P in the tensor-core path): close, not equal.
    assert (outs[0] - outs[1]).abs().max().item() < 5e-3
