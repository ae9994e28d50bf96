"""GPU parity: FP8 (E4M3) KV cache. The quantising write is bit-exact against the
oracle (codes and scales); decode over the FP8 cache matches the fp64 oracle run on
the dequantised cache, within the decode tolerance."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp8_ref as f8
from oracle import paged_ref as ref
from paged_kv_cache_77_gb300 import api
from tests.gpu_cases import DecodeCase, compare, oracle_fp8_all

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["gqa_long"]


class Fp8Case:
    """A DecodeCase whose cache is quantised to FP8 on the GPU (checked bit for bit
    against the oracle's own quantisation), with the new rows then written by the
    FP8 write and the tails of the last blocks poisoned with NaN codes and scales."""

    def __init__(self, wl, d=None, check_rows=None, whole=False, base=None):
        """``whole``: the oracle's side is left to ``oracle_fp8_all`` (per sequence, in
        a process pool), which gets host copies of the codes and scales taken here
        right after the GPU's writes; only the GPU's tails are poisoned. ``base``: a
        DecodeCase of (wl, d) prepared by the caller, used in place of a fresh one."""
        self.base = base if base is not None else DecodeCase(wl, d, poison=True)
        c, wl = self.base, self.base.wl
        nb, bs, hkv, dh = c.v["k_cache"].shape
        self.nb, self.bs, self.hkv = nb, bs, hkv
        dev = "cuda"
        self.kc = torch.empty((nb, bs, hkv, dh), dtype=torch.uint8, device=dev)
        self.vc = torch.empty_like(self.kc)
        self.ks = torch.empty((nb, hkv, bs), dtype=torch.float32, device=dev)
        self.vs = torch.empty_like(self.ks)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        every = torch.arange(nb * bs, dtype=torch.int32, device=dev)
        api.kv_cache_write_fp8(self.kc, self.vc, self.ks, self.vs, c.v["k_cache"].view(nb * bs, hkv, dh),
                               c.v["v_cache"].view(nb * bs, hkv, dh), every, dev_status=self.status)
        api.kv_cache_write_fp8(self.kc, self.vc, self.ks, self.vs, c.v["k_new"], c.v["v_new"], c.slots,
                               dev_status=self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        if whole:
            self.gpu_codes = {"kc": self.kc.cpu().numpy(), "ks": self.ks.cpu().numpy(),
                              "vc": self.vc.cpu().numpy(), "vs": self.vs.cpu().numpy()}
            self.codes = None
            self._poison_tails()
            return
        # The oracle quantises the same bf16 rows (blocks in `check_rows`' tables, or all
        # but the NaN-poisoned null block) and applies the same write.
        blocks = self._blocks(check_rows)
        kb, vb = c.pre["k_cache"], c.pre["v_cache"]
        self.codes = {}
        for name, pre, new, cc, sc in (("k", kb, c.v["k_new"], self.kc, self.ks),
                                       ("v", vb, c.v["v_new"], self.vc, self.vs)):
            codes = np.zeros((nb, bs, hkv, dh), np.uint8)
            scales = np.zeros((nb, hkv, bs), np.float32)
            q, s = f8.quantize_rows(pre[blocks])
            codes[blocks], scales[blocks] = q, s.transpose(0, 2, 1)
            keep = np.isin(c.slots_np // bs, blocks)
            codes, scales = f8.cache_write_fp8(codes, scales, synth.bf16_bits(new)[keep], c.slots_np[keep])
            idx = torch.from_numpy(blocks).cuda()
            got_c, got_s = cc[idx].cpu().numpy(), sc[idx].cpu().numpy()
            assert np.array_equal(got_c, codes[blocks]), f"{name} codes differ from the oracle"
            assert np.array_equal(got_s, scales[blocks]), f"{name} scales differ from the oracle"
            self.codes[name] = (codes, scales)
        self._poison_tails()

    def _blocks(self, rows):
        c = self.base
        if rows is None:
            return np.arange(1, self.nb)
        used = set()
        for b in rows:
            n = -(-int(c.d.seq_lens[b]) // self.bs)
            used.update(int(x) for x in c.table_np[b, :n])
        used.discard(0)
        return np.array(sorted(used), dtype=np.int64)

    def _poison_tails(self):
        # Positions past each sequence's length in its last block: NaN codes and
        # scales, on the GPU and in the oracle's copies (which never read them).
        c = self.base
        for b, n in enumerate(c.d.seq_lens):
            n = int(n)
            if n % self.bs == 0 or n == 0:
                continue
            blk = int(c.table_np[b, n // self.bs])
            off = n % self.bs
            for cc, sc in ((self.kc, self.ks), (self.vc, self.vs)):
                cc[blk, off:] = 0x7F
                sc[blk, :, off:] = float("nan")
            for name in (("k", "v") if self.codes is not None else ()):
                codes, scales = self.codes[name]
                codes[blk, off:] = 0x7F
                scales[blk, :, off:] = np.nan

    def run(self, rows, out_dtype=torch.float32):
        c, wl = self.base, self.base.wl
        lse = torch.full((wl.batch, wl.num_heads), float("nan"), device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = api.paged_attention_decode_fp8(c.v["q"], self.kc, self.vc, self.ks, self.vs, c.table,
                                             c.seq_lens, wl.scale, wl.window, lse=lse,
                                             out_dtype=out_dtype, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        kdq = f8.dequantize_cache(*self.codes["k"])
        vdq = f8.dequantize_cache(*self.codes["v"])
        q64 = c.v["q"].double().cpu().numpy()
        o_ref, lse_ref = ref.paged_decode(q64, kdq, vdq, c.table_np, c.d.seq_lens, wl.block_size,
                                          wl.scale, wl.window, batch_indices=rows)
        return out, lse, o_ref, lse_ref


@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (32, 2)])
@pytest.mark.parametrize("window", [0, 200])
def test_fp8_decode_small_edge_cases(H, Hkv, window):
    lens = [1, 127, 128, 129, 700, 0, 2000, 255]
    wl = BASE.scaled(batch=len(lens), num_heads=H, num_kv_heads=Hkv, window=window, seed=17)
    case = Fp8Case(wl, synth.draw_explicit(wl, lens))
    rows = list(range(len(lens)))
    out, lse, o_ref, lse_ref = case.run(rows)
    compare(out, lse, o_ref, lse_ref, rows, f"fp8 H{H}/Hkv{Hkv}/W{window}")
    assert out[5].abs().max().item() == 0.0 and torch.isinf(lse[5]).all()


def test_fp8_decode_bf16_output_and_many_splits():
    lens = [5000, 3, 4096, 12000]
    wl = BASE.scaled(batch=4, num_heads=64, num_kv_heads=8, seed=18)
    case = Fp8Case(wl, synth.draw_explicit(wl, lens))
    out, lse, o_ref, lse_ref = case.run([0, 1, 2, 3], out_dtype=torch.bfloat16)
    compare(out, lse, o_ref, lse_ref, [0, 1, 2, 3], "fp8 bf16 out")


def test_fp8_write_zero_rows_and_bad_slot():
    nb, bs, hkv = 3, 128, 2
    kc = torch.zeros((nb, bs, hkv, 128), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.full((nb, hkv, bs), 7.0, device="cuda")
    vs = torch.full_like(ks, 7.0)
    g = torch.Generator().manual_seed(19)
    k = torch.randn((4, hkv, 128), generator=g).to(torch.bfloat16)
    k[1] = 0
    v = torch.randn((4, hkv, 128), generator=g).to(torch.bfloat16)
    slots = torch.tensor([5, 6, -1, nb * bs + 1], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.kv_cache_write_fp8(kc, vc, ks, vs, k.cuda(), v.cuda(), slots.cuda(), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 1  # PKV_DEV_BAD_SLOT
    want_c, want_s = f8.cache_write_fp8(np.zeros((nb, bs, hkv, 128), np.uint8),
                                        np.full((nb, hkv, bs), 7.0, np.float32),
                                        synth.bf16_bits(k[:2]), np.array([5, 6]))
    assert np.array_equal(kc.cpu().numpy(), want_c)
    assert np.array_equal(ks.cpu().numpy(), want_s)
    assert ks[0, :, 6].abs().max().item() == 0.0  # the all-zero row: scale 0


@pytest.mark.parametrize("name", ["gqa_long", "swa"])
def test_fp8_decode_workloads_full_size(name):
    # Every sequence: each pool task quantises the sequence's blocks of the bf16 cache
    # and applies its quantising write with the oracle, counts codes and scales that
    # differ from the GPU's (bit for bit), and decodes over the dequantised blocks.
    wl = synth.WORKLOADS[name]
    case = Fp8Case(wl, synth.draw(wl), whole=True)
    c = case.base
    lse = torch.full((wl.batch, wl.num_heads), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.paged_attention_decode_fp8(c.v["q"], case.kc, case.vc, case.ks, case.vs, c.table,
                                         c.seq_lens, wl.scale, wl.window, lse=lse, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, lse_ref, mismatches = oracle_fp8_all(c, case.gpu_codes)
    assert mismatches == 0, f"{mismatches} FP8 codes or scales differ from the oracle's"
    rows = list(range(wl.batch))
    mx, mean = compare(out, lse, o_ref, lse_ref, rows, f"fp8 {name}")
    print(f"fp8 {name}: {len(rows)} of {wl.batch} sequences, max abs {mx:.2e} mean abs {mean:.2e}")
