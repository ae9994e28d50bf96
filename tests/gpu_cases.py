"""Shared set-up of GPU parity cases: draw inputs, build tables with the library's
host generator (checked against the oracle's), write through the CUDA path and
through the oracle, and compare."""
from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import block_pool_ref as bp
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api

MAX_ABS_TOL = 1e-2  # attention outputs from bf16 inputs vs the fp64 oracle
MEAN_ABS_TOL = 1e-3
LSE_TOL = 2e-3
# The prefill kernel's log-sum-exp is taken from the sum of the bf16-rounded weights
# that its output uses (the output is then an exact convex combination of V rows).
# Round-to-nearest-even to bf16's 8 significant bits moves each weight by at most 2^-8
# of itself, so the sum too, and its log by at most ln(1 + 2^-8) = 3.9e-3 (reached
# when one key dominates a row); the scores' own fp32 error comes on top.
PREFILL_LSE_TOL = 4e-3 + 5e-4


def tables(wl: synth.Workload, d: synth.Draw):
    """Library block table + slot mapping, asserted equal to the oracle's."""
    if wl.layout == "arange":
        table = api.build_block_table_arange(wl.batch, d.max_blocks_per_seq)
        ref_table = bp.block_table_arange(wl.batch, d.max_blocks_per_seq)
    else:
        # Speculative decode keeps blocks live from the first new row's window start.
        win = wl.window + wl.q_hi - 1 if wl.kind == "spec_decode" and wl.window > 0 else wl.window
        table = api.BlockPool(d.num_blocks, d.pool_order).build_block_table(
            d.seq_lens, wl.block_size, win, d.max_blocks_per_seq)
        ref_table = bp.prepare_block_tables(bp.BlockPool(d.num_blocks, d.pool_order), d.seq_lens,
                                            wl.block_size, win, d.max_blocks_per_seq)
    assert np.array_equal(table, ref_table)
    slots = api.build_slot_mapping(table, d.start_pos, d.num_new, wl.block_size)
    assert np.array_equal(slots, bp.slot_mapping(ref_table, d.start_pos, d.num_new, wl.block_size))
    return table, slots


class DecodeCase:
    """One decode instance on the GPU plus the oracle's view of the same bytes."""

    def __init__(self, wl: synth.Workload, d: synth.Draw | None = None, poison: bool = True):
        self.wl = wl
        self.d = d if d is not None else synth.draw(wl)
        self.v = synth.values(wl, self.d, "cuda", poison_null=poison)
        self.table_np, self.slots_np = tables(wl, self.d)
        self.table = torch.from_numpy(self.table_np).cuda()
        self.slots = torch.from_numpy(self.slots_np).cuda()
        self.seq_lens = torch.from_numpy(self.d.seq_lens).cuda()
        names = ("cache_nope", "cache_rope") if wl.kind == "mla_decode" else ("k_cache", "v_cache")
        # Host copies taken before the CUDA write: the oracle writes its own.
        self.pre = {n: synth.bf16_bits(self.v[n]) for n in names}
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def gpu_write(self):
        if self.wl.kind == "mla_decode":
            api.kv_cache_write(self.v["cache_nope"], self.v["cache_rope"], self.v["nope_new"],
                               self.v["rope_new"], self.slots, dev_status=self.status)
        else:
            api.kv_cache_write(self.v["k_cache"], self.v["v_cache"], self.v["k_new"],
                               self.v["v_new"], self.slots, dev_status=self.status)

    def oracle_write(self):
        if self.wl.kind == "mla_decode":
            pairs = (("cache_nope", "nope_new"), ("cache_rope", "rope_new"))
        else:
            pairs = (("k_cache", "k_new"), ("v_cache", "v_new"))
        self.post = {c: ref.cache_write(self.pre[c], synth.bf16_bits(self.v[r]), self.slots_np)
                     for c, r in pairs}

    def poison_tails(self):
        """NaN in every cache row past a sequence's length inside its last block, on
        the GPU and in the oracle's copy (which never reads them). Such rows hold
        whatever the memory held before; attention must not depend on them."""
        bs = self.wl.block_size
        names = list(self.post)
        for b, n in enumerate(self.d.seq_lens):
            n = int(n)
            if n == 0 or n % bs == 0:
                continue
            blk, off = int(self.table_np[b, n // bs]), n % bs
            for name in names:
                self.v[name][blk, off:] = float("nan")
                self.post[name][blk, off:] = synth.BF16_NAN_BITS

    def check_write_bit_exact(self):
        for name, expect in self.post.items():
            got = synth.bf16_bits(self.v[name])
            assert np.array_equal(got, expect), f"{name} differs from the oracle's write"
        assert int(self.status.item()) == 0


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) at |x|."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.ldexp(1.0, np.floor(np.log2(ax)).astype(np.int64) - 8)


def compare(out: torch.Tensor, lse: torch.Tensor | None, o_ref: np.ndarray, lse_ref: np.ndarray,
            rows, what: str, lse_tol: float = LSE_TOL):
    """Max / mean abs error on the selected leading-index rows.

    A bf16 output is the kernel's fp32 result rounded to nearest even, so each element
    may differ from the exact value by the 1e-2 bound plus half a bf16 ulp (0.0156 at
    |o| in [4, 8)); fp32 outputs are held to the bound itself.
    """
    got = out.float().cpu().numpy()[rows]
    exp = o_ref[rows]
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - exp)
    if out.dtype == torch.bfloat16:
        excess = err - bf16_half_ulp(np.abs(exp) + MAX_ABS_TOL)
        assert excess.max() <= MAX_ABS_TOL, f"{what}: max abs err beyond bf16 rounding {excess.max():.3e}"
    else:
        assert err.max() <= MAX_ABS_TOL, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS_TOL, f"{what}: mean abs err {err.mean():.3e}"
    if lse is not None:
        lg = lse.cpu().numpy()[rows]
        le = lse_ref[rows]
        fin = np.isfinite(le)
        assert np.array_equal(np.isfinite(lg), fin)
        dl = np.abs(lg[fin] - le[fin]).max(initial=0)
        assert dl <= lse_tol, f"{what}: lse error {dl:.3e} (|lse| up to {np.abs(le[fin]).max(initial=0):.1f})"
    return float(err.max()), float(err.mean())


# ------------------------------------------------------------------ whole-batch oracle
# Full-size parity compares every row of a workload. The unchanged oracle runs once
# per sequence (or per run of query rows of one sequence) in a spawn process pool on
# the host's cores; the caches reach the workers as memory-mapped files.
def _pool_run(shared: dict, tasks: list, costs):
    from oracle.pool import OraclePool

    order = np.argsort(-np.asarray(costs, dtype=np.float64), kind="stable")
    with OraclePool(shared) as pool:
        res = pool.map([tasks[i] for i in order])
    out = [None] * len(tasks)
    for k, i in enumerate(order):
        out[i] = res[k]
    print(f"oracle: {len(tasks)} parts on {pool.workers} processes in {pool.seconds:.1f} s")
    return out


def oracle_decode_all(case: DecodeCase, window: int | None = None):
    """(o, lse) of the oracle for every sequence of a decode or speculative-decode case,
    on the caches after the oracle's write (case.post)."""
    from oracle.pool import task

    wl = case.wl
    window = wl.window if window is None else window
    q64 = case.v["q"].double().cpu().numpy()
    fn = "paged_spec_decode" if wl.kind == "spec_decode" else "paged_decode"
    shared = {"k": case.post["k_cache"], "v": case.post["v_cache"]}
    tasks = [task(fn, shared_kwargs={"k_cache": "k", "v_cache": "v"}, q=q64[b:b + 1],
                  block_table=case.table_np[b:b + 1], seq_lens=case.d.seq_lens[b:b + 1],
                  block_size=wl.block_size, scale=wl.scale, window=window)
             for b in range(wl.batch)]
    res = _pool_run(shared, tasks, case.d.seq_lens)
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def oracle_mla_all(case: DecodeCase):
    """(o, lse) of the oracle for every sequence of an MLA case (one or q_len rows)."""
    from oracle.pool import task

    wl = case.wl
    qn = case.v["q_nope"].double().cpu().numpy()
    qr = case.v["q_rope"].double().cpu().numpy()
    fn = "mla_spec_decode" if qn.ndim == 4 else "mla_decode"
    shared = {"nope": case.post["cache_nope"], "rope": case.post["cache_rope"]}
    tasks = [task(fn, shared_kwargs={"cache_nope": "nope", "cache_rope": "rope"},
                  q_nope=qn[b:b + 1], q_rope=qr[b:b + 1], block_table=case.table_np[b:b + 1],
                  seq_lens=case.d.seq_lens[b:b + 1], block_size=wl.block_size, scale=wl.scale)
             for b in range(wl.batch)]
    res = _pool_run(shared, tasks, case.d.seq_lens)
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def oracle_prefill_all(case: DecodeCase, causal: bool = True, rows_per_part: int = 64):
    """(o, lse) of the oracle for every query row of a prefill case.

    Rows [r0, r1) of a sequence with c prior keys and q new rows form the prefill
    problem with c + r0 prior keys and r1 - r0 new rows under the bottom-right mask:
    row r0 + i sees keys j <= c + r0 + i in both. Without the causal mask every row
    sees all len keys, so the part keeps the sequence's length."""
    from oracle.pool import task

    wl = case.wl
    q64 = case.v["q"].double().cpu().numpy()
    shared = {"k": case.post["k_cache"], "v": case.post["v_cache"]}
    tasks, costs = [], []
    begin = 0
    for b in range(wl.batch):
        qlen, n = int(case.d.num_new[b]), int(case.d.seq_lens[b])
        c = n - qlen
        for r0 in range(0, qlen, rows_per_part):
            r1 = min(qlen, r0 + rows_per_part)
            kv = c + r1 if causal else n
            tasks.append(task("paged_prefill", shared_kwargs={"k_cache": "k", "v_cache": "v"},
                              q=q64[begin + r0:begin + r1], cu_seqlens_q=np.array([r1 - r0]),
                              block_table=case.table_np[b:b + 1], seq_lens_kv=np.array([kv]),
                              block_size=wl.block_size, scale=wl.scale, causal=causal))
            costs.append((r1 - r0) * kv)
        begin += qlen
    res = _pool_run(shared, tasks, costs)
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def oracle_fp8_all(base: DecodeCase, codes: dict):
    """(o, lse, mismatches) of the oracle for every sequence of an FP8 decode case.

    ``codes`` holds host copies of the GPU's FP8 cache right after its writes (before
    any poisoning): {"kc", "ks", "vc", "vs"}. Each worker quantises the sequence's
    blocks of the bf16 cache, applies the sequence's quantising write, counts entries
    that differ from the GPU's, and decodes over the dequantised blocks."""
    from oracle.pool import task

    wl = base.wl
    q64 = base.v["q"].double().cpu().numpy()
    shared = {"kp": base.pre["k_cache"], "vp": base.pre["v_cache"], **codes}
    kn, vn = synth.bf16_bits(base.v["k_new"]), synth.bf16_bits(base.v["v_new"])
    ends = np.cumsum(base.d.num_new)
    starts = ends - base.d.num_new
    tasks = [task("fp8_sequence", module="tests.oracle_tasks",
                  shared_kwargs={"k_pre": "kp", "v_pre": "vp", "gpu_kc": "kc", "gpu_ks": "ks",
                                 "gpu_vc": "vc", "gpu_vs": "vs"},
                  q_row=q64[b:b + 1], table_row=base.table_np[b], seq_len=int(base.d.seq_lens[b]),
                  slots=base.slots_np[starts[b]:ends[b]], k_new=kn[starts[b]:ends[b]],
                  v_new=vn[starts[b]:ends[b]], block_size=wl.block_size, scale=wl.scale,
                  window=wl.window)
             for b in range(wl.batch)]
    res = _pool_run(shared, tasks, base.d.seq_lens)
    return (np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res]),
            sum(r[2] for r in res))
