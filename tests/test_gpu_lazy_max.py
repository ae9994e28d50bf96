"""GPU parity when later key blocks beat the running reference max.

Every attention kernel keeps, per query row (or column), a reference max that it
raises only when a tile's max beats it by more than 8 in log2 units, and then
rescales the output accumulated so far. With keys drawn N(0,1) the first tile
almost always sets a reference that no later tile beats by 8, so that path would go
untested at the workloads. Here the keys of logical block i of every sequence (and
the new rows written into it) are multiplied by 1 + 1.5 min(i, 8): the scores grow
along the first blocks of every sequence and later tiles raise the reference again
and again. Each case first
counts, on the oracle's fp64 scores and with the kernels' tile sizes, the tiles that
raise it (the count must be positive), then compares the GPU with the oracle. The
sequences are long enough that a CTA's range holds several tiles of one sequence, so
the raise happens inside a kernel's pieces and not only across the merge. Values are
left N(0,1): for MLA, whose value is the latent row, only the rope part grows.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import PREFILL_LSE_TOL, DecodeCase, compare
from tests import test_gpu_decode as tdec
from tests import test_gpu_fp8 as tfp8
from tests import test_gpu_mla as tmla
from tests import test_gpu_prefill as tpf
from tests import test_gpu_spec as tspec

pytestmark = pytest.mark.gpu

LOG2E = 1.0 / np.log(2.0)


def _growth(i):
    # Capped, so that the scores stay within ~50 log2 units: beyond, the fp32 rounding
    # of the scores themselves (relative) would dominate the log-sum-exp's error.
    return 1.0 + 1.5 * min(i, 8)


def grow(case: DecodeCase, caches, rows):
    """Scale block i of every sequence by _growth(i) in `caches` (GPU and the oracle's
    host copy; blocks used by one sequence only) and each new row in `rows` by the
    factor of the block it is written into."""
    bs = case.wl.block_size
    owner = {}
    for b, n in enumerate(case.d.seq_lens):
        for i in range(-(-int(n) // bs)):
            blk = int(case.table_np[b, i])
            owner[blk] = None if blk in owner else (b, i)
    for blk, who in owner.items():
        if who is None:
            continue
        f = _growth(who[1])
        for name in caches:
            t = case.v[name]
            t[blk] = (t[blk].float() * f).to(torch.bfloat16)
    t = 0
    for b in range(case.wl.batch):
        for k in range(int(case.d.num_new[b])):
            f = _growth((int(case.d.start_pos[b]) + k) // bs)
            for name in rows:
                case.v[name][t] = (case.v[name][t].float() * f).to(torch.bfloat16)
            t += 1
    for name in caches:
        case.pre[name] = synth.bf16_bits(case.v[name])


def raises(z, tile):
    """Tiles after the first whose max beats the running reference by more than 8
    (z: one row's scores in log2 units, in key order)."""
    m, n = -np.inf, 0
    for t0 in range(0, len(z), tile):
        mt = z[t0:t0 + tile].max()
        if mt > m + 8.0:
            n += m > -np.inf
            m = mt
    return n


def decode_raises(case, tile, q_rows=None):
    """Raise count summed over (sequence, head) on the oracle's post-write cache."""
    wl, total = case.wl, 0
    q = case.v["q"].double().cpu().numpy()
    n_rep = wl.num_heads // wl.num_kv_heads
    for b, n in enumerate(case.d.seq_lens):
        K = ref.gather_sequence(case.post["k_cache"], case.table_np[b], int(n), wl.block_size)
        qb = q[b] if q_rows is None else q[b, q_rows]
        for h in range(wl.num_heads):
            z = wl.scale * LOG2E * (K[:, h // n_rep] @ qb[h])
            total += raises(z, tile)
    return total


@pytest.mark.parametrize("kernel", list(tdec.KERNELS))
@pytest.mark.parametrize("H,Hkv,window", [(32, 8, 0), (8, 8, 0), (32, 4, 4000)])
def test_decode_with_growing_keys(kernel, H, Hkv, window):
    api.set_decode_kernel(tdec.KERNELS[kernel])
    try:
        lens = [6000, 129, 9000, 700, 1] if window == 0 else [8000] * 6 + [129, 700]
        wl = tdec.BASE.scaled(batch=len(lens), num_heads=H, num_kv_heads=Hkv, window=window,
                              seed=61)
        case = DecodeCase(wl, synth.draw_explicit(wl, lens))
        grow(case, ["k_cache"], ["k_new"])
        rows = list(range(len(lens)))
        out, lse, o_ref, lse_ref = tdec._run_decode(case, rows)
        assert decode_raises(case, 128) > 0
        compare(out, lse, o_ref, lse_ref, rows, f"{kernel} growing keys H{H}/Hkv{Hkv}/W{window}")
    finally:
        api.set_decode_kernel(api.KERNEL_AUTO)


def test_spec_decode_with_growing_keys():
    lens = [12000, 9000, 260, 3000]
    case = tspec._lens_case(32, 4, 4, 0, lens, 62)
    grow(case, ["k_cache"], ["k_new"])
    rows = list(range(len(lens)))
    out, lse, o_ref, lse_ref = tspec._run(case, rows)
    assert decode_raises(case, 128, q_rows=-1) > 0
    compare(out, lse, o_ref, lse_ref, rows, "spec decode growing keys")


def test_fp8_decode_with_growing_keys():
    lens = [9000, 129, 12000, 700]
    wl = tfp8.BASE.scaled(batch=len(lens), num_heads=32, num_kv_heads=4, seed=63)
    d = synth.draw_explicit(wl, lens)
    base = DecodeCase(wl, d, poison=True)
    grow(base, ["k_cache"], ["k_new"])
    case = tfp8.Fp8Case(wl, d, base=base)
    rows = list(range(len(lens)))
    out, lse, o_ref, lse_ref = case.run(rows)
    base.oracle_write()
    assert decode_raises(base, 128) > 0
    compare(out, lse, o_ref, lse_ref, rows, "fp8 growing keys")


@pytest.mark.parametrize("H", [128, 16])
def test_mla_with_growing_keys(H):
    lens = [8192, 8000, 6000, 3000, 65, 900, 129]
    wl = tmla.MLA.scaled(batch=len(lens), num_heads=H, seed=64)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens))
    grow(case, ["cache_rope"], ["rope_new"])
    rows = list(range(len(lens)))
    out, lse, o_ref, lse_ref = tmla._run(case, rows)
    qn = case.v["q_nope"].double().cpu().numpy()
    qr = case.v["q_rope"].double().cpu().numpy()
    total = 0
    for b, n in enumerate(case.d.seq_lens):
        N = ref.gather_sequence(case.post["cache_nope"], case.table_np[b], int(n), wl.block_size)[:, 0]
        R = ref.gather_sequence(case.post["cache_rope"], case.table_np[b], int(n), wl.block_size)[:, 0]
        for h in range(H):
            total += raises(wl.scale * LOG2E * (N @ qn[b, h] + R @ qr[b, h]), 64)
    assert total > 0
    compare(out, lse, o_ref, lse_ref, rows, f"mla growing keys H{H}")


def test_prefill_with_growing_keys():
    prior, qlen = [6000, 0, 3000], [64, 200, 1]
    wl = tpf.MIX.scaled(batch=len(prior), seed=65)
    case = tpf._case(wl, prior, qlen)
    grow(case, ["k_cache"], ["k_new"])
    T = int(sum(qlen))
    rows = list(range(T))
    out, lse, o_ref, lse_ref = tpf._run(case, rows)
    # The last query row of the first sequence sees its whole prior context.
    q = case.v["q"].double().cpu().numpy()
    n0 = prior[0] + qlen[0]
    K = ref.gather_sequence(case.post["k_cache"], case.table_np[0], n0, wl.block_size)
    n_rep = wl.num_heads // wl.num_kv_heads
    total = sum(raises(wl.scale * LOG2E * (K[:, h // n_rep] @ q[qlen[0] - 1, h]), 128)
                for h in range(wl.num_heads))
    assert total > 0
    compare(out, lse, o_ref, lse_ref, rows, "prefill growing keys", lse_tol=PREFILL_LSE_TOL)
