"""GPU parity on seeded random configurations of every attention entry point.

The other GPU tests pick their shapes by hand (edges, the workloads). Here each case
draws a batch size, head layout, lengths (including 0, 1 and block edges), window,
number of new rows and output type from a seeded generator, runs the CUDA path and
compares every row with the oracle, under the same bounds as the rest of the suite.
"""
import numpy as np
import pytest
import torch

import synth
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import PREFILL_LSE_TOL, DecodeCase, compare
from tests import test_gpu_decode as tdec
from tests import test_gpu_fp8 as tfp8
from tests import test_gpu_mla as tmla
from tests import test_gpu_mla_spec as tmspec
from tests import test_gpu_prefill as tpf
from tests import test_gpu_spec as tspec

pytestmark = pytest.mark.gpu

N_CASES = 6
EDGE_LENS = [0, 1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257]


def _lens(rng, B, hi, lo=0):
    """Mix of block-edge lengths and uniform draws."""
    out = []
    for _ in range(B):
        if rng.random() < 0.4:
            out.append(int(rng.choice([x for x in EDGE_LENS if lo <= x <= hi])))
        else:
            out.append(int(rng.integers(lo, hi + 1)))
    return out


def _heads(rng, max_rep=16):
    n_rep = int(rng.choice([r for r in (1, 2, 4, 8, 16) if r <= max_rep]))
    hkv = int(rng.choice([1, 2, 4, 8]))
    while n_rep * hkv > 64:
        hkv //= 2
    return n_rep * hkv, hkv


@pytest.mark.parametrize("case_id", range(N_CASES))
def test_fuzz_decode(case_id):
    rng = np.random.default_rng(7000 + case_id)
    B = int(rng.integers(1, 10))
    H, Hkv = _heads(rng)
    window = int(rng.choice([0, 0, int(rng.integers(1, 600))]))
    lens = _lens(rng, B, 3000)
    kernel = list(tdec.KERNELS)[case_id % 2]
    out_dtype = torch.bfloat16 if rng.random() < 0.5 else torch.float32
    wl = tdec.BASE.scaled(batch=B, num_heads=H, num_kv_heads=Hkv, window=window,
                          seed=7000 + case_id)
    api.set_decode_kernel(tdec.KERNELS[kernel])
    try:
        case = DecodeCase(wl, synth.draw_explicit(wl, lens))
        rows = list(range(B))
        out, lse, o_ref, lse_ref = tdec._run_decode(case, rows, out_dtype=out_dtype)
        compare(out, lse, o_ref, lse_ref, rows,
                f"{kernel} B{B} H{H}/{Hkv} W{window} lens {lens} {out_dtype}")
    finally:
        api.set_decode_kernel(api.KERNEL_AUTO)


@pytest.mark.parametrize("case_id", range(N_CASES))
def test_fuzz_spec_decode(case_id):
    rng = np.random.default_rng(7100 + case_id)
    Q = int(rng.integers(1, 5))
    n_rep = int(rng.choice([r for r in (1, 2, 4, 8) if r * Q <= 32]))
    Hkv = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 8))
    window = int(rng.choice([0, int(rng.integers(4, 500))]))
    lens = _lens(rng, B, 2500, lo=1)
    case = tspec._lens_case(n_rep * Hkv, Hkv, Q, window, lens, 7100 + case_id)
    rows = list(range(B))
    out, lse, o_ref, lse_ref = tspec._run(case, rows)
    compare(out, lse, o_ref, lse_ref, rows, f"spec B{B} Q{Q} H{n_rep * Hkv}/{Hkv} W{window} lens {lens}")


@pytest.mark.parametrize("case_id", range(N_CASES))
def test_fuzz_fp8_decode(case_id):
    rng = np.random.default_rng(7200 + case_id)
    B = int(rng.integers(1, 8))
    H, Hkv = _heads(rng, max_rep=8)
    window = int(rng.choice([0, int(rng.integers(1, 600))]))
    lens = _lens(rng, B, 3000)
    wl = tfp8.BASE.scaled(batch=B, num_heads=H, num_kv_heads=Hkv, window=window, seed=7200 + case_id)
    case = tfp8.Fp8Case(wl, synth.draw_explicit(wl, lens))
    rows = list(range(B))
    out, lse, o_ref, lse_ref = case.run(rows)
    compare(out, lse, o_ref, lse_ref, rows, f"fp8 B{B} H{H}/{Hkv} W{window} lens {lens}")


@pytest.mark.parametrize("case_id", range(N_CASES))
def test_fuzz_mla(case_id):
    rng = np.random.default_rng(7300 + case_id)
    B = int(rng.integers(1, 8))
    H = int(rng.choice([8, 16, 40, 128]))
    lens = _lens(rng, B, 2500)
    out_dtype = torch.bfloat16 if rng.random() < 0.5 else torch.float32
    wl = tmla.MLA.scaled(batch=B, num_heads=H, seed=7300 + case_id)
    case = DecodeCase(wl, synth.draw_explicit(wl, lens))
    rows = list(range(B))
    out, lse, o_ref, lse_ref = tmla._run(case, rows, out_dtype=out_dtype)
    compare(out, lse, o_ref, lse_ref, rows, f"mla B{B} H{H} lens {lens} {out_dtype}")


@pytest.mark.parametrize("case_id", range(N_CASES))
def test_fuzz_mla_spec(case_id):
    rng = np.random.default_rng(7400 + case_id)
    Q = int(rng.integers(2, 5))  # one row per sequence is the plain MLA decode above
    B = int(rng.integers(1, 6))
    H = int(rng.choice([16, 64, 128]))
    lens = _lens(rng, B, 2000)
    case = tmspec._case(Q, H, lens, 7400 + case_id)
    rows = list(range(B))
    out, lse, o_ref, lse_ref = tmspec._run(case, rows)
    compare(out, lse, o_ref, lse_ref, rows, f"mla spec B{B} Q{Q} H{H} lens {lens}")


@pytest.mark.parametrize("case_id", range(N_CASES))
def test_fuzz_prefill(case_id):
    rng = np.random.default_rng(7500 + case_id)
    B = int(rng.integers(1, 6))
    H, Hkv = _heads(rng)
    prior = _lens(rng, B, 1500)
    qlen = [int(x) for x in rng.choice([0, 1, 2, 31, 32, 33, 127, 128, 129, 300], size=B)]
    causal = bool(rng.random() < 0.8)
    wl = tpf.MIX.scaled(batch=B, num_heads=H, num_kv_heads=Hkv, seed=7500 + case_id)
    case = tpf._case(wl, prior, qlen)
    T = int(sum(qlen))
    rows = list(range(T))
    out, lse, o_ref, lse_ref = tpf._run(case, rows, causal=causal)
    if T:
        compare(out, lse, o_ref, lse_ref, rows,
                f"prefill B{B} H{H}/{Hkv} prior {prior} q {qlen} causal {causal}",
                lse_tol=PREFILL_LSE_TOL)
