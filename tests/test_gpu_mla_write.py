"""GPU parity: fused MLA cache write (RMSNorm + RoPE + slot write) vs the fp64 oracle.

The GPU computes in fp32, the oracle in fp64; both round to bf16 to nearest even.
The two can land on different sides of a rounding boundary only when the exact
value lies within fp32 rounding distance of it, so results may differ by one bf16
unit in the last place on rare elements. The RoPE sum x*cos + x'*sin can cancel;
its fp32 error is bounded by the operands (about 2^-23 (|x cos| + |x' sin|)), not by
the result, so a rope element may also differ by up to 2^-20 times the largest
rope input of its row. The bar: every element within those bounds, at least
99.9 % bit-identical on samples of 10,000 elements or more, rows not written
bit-identical to before."""
import numpy as np
import pytest
import torch

import synth
from oracle import mla_write_ref as mw
from oracle.paged_ref import bf16_bits_to_f64
from paged_kv_cache_77_gb300 import api

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _rope_floor(latent_bits):
    """Per-row cancellation allowance of the rope sum: 2^-20 * max |rope input|."""
    r = np.abs(bf16_bits_to_f64(latent_bits[:, 512:]))
    return (2.0 ** -20) * r.max(axis=1, keepdims=True)


def _ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 units between same-sign finite bit patterns (sign-magnitude)."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(key(a_bits) - key(b_bits))


def _check(got, want, what, abs_floor=None):
    d = _ulp_diff(got, want)
    ok = d <= 1
    if abs_floor is not None:
        diff = np.abs(bf16_bits_to_f64(got) - bf16_bits_to_f64(want))
        ok |= diff <= abs_floor
    assert ok.all(), f"{what}: {int(d[~ok].max())} ulp beyond the bound"
    exact = float((d == 0).mean())
    if d.size >= 10000:  # the fraction means something only on a large sample
        assert exact >= 0.999, f"{what}: only {exact:.5f} bit-identical"
    return exact


def _run(T, nb, seed, neg=0, outputs=True):
    v = synth.draw_mla_write(T, nb, seed, device="cuda", neg_slots=neg)
    pre_n, pre_r = synth.bf16_bits(v["cache_nope"]), synth.bf16_bits(v["cache_rope"])
    kn = torch.empty((T, 512), dtype=torch.bfloat16, device="cuda") if outputs else None
    kr = torch.empty((T, 64), dtype=torch.bfloat16, device="cuda") if outputs else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_rmsnorm_rope_write(v["cache_nope"], v["cache_rope"], v["latent"], v["gamma"], v["cos"],
                               v["sin"], v["slots"], EPS, k_nope_out=kn, k_rope_out=kr, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return v, pre_n, pre_r, kn, kr


@pytest.mark.parametrize("T", [1, 7, 1000, 4099])
def test_fused_write_matches_oracle(T):
    nb = max(4, (T + 127) // 128 + 3)
    v, pre_n, pre_r, kn, kr = _run(T, nb, 81 + T, neg=min(3, T // 3))
    slots = v["slots"].cpu().numpy()
    post_n, post_r, nope, rope = mw.mla_rmsnorm_rope_write(
        pre_n, pre_r, synth.bf16_bits(v["latent"]), synth.bf16_bits(v["gamma"]),
        v["cos"].cpu().numpy(), v["sin"].cpu().numpy(), slots, 512, EPS)
    _check(synth.bf16_bits(kn), nope, "k_nope")
    floor = _rope_floor(synth.bf16_bits(v["latent"]))
    _check(synth.bf16_bits(kr), rope, "k_rope", floor)
    got_n, got_r = synth.bf16_bits(v["cache_nope"]), synth.bf16_bits(v["cache_rope"])
    written = np.zeros(nb * 128, dtype=bool)
    written[slots[slots >= 0]] = True
    flat_gn, flat_pn = got_n.reshape(nb * 128, -1), post_n.reshape(nb * 128, -1)
    flat_gr, flat_pr = got_r.reshape(nb * 128, -1), post_r.reshape(nb * 128, -1)
    assert np.array_equal(flat_gn[~written], pre_n.reshape(nb * 128, -1)[~written])
    assert np.array_equal(flat_gr[~written], pre_r.reshape(nb * 128, -1)[~written])
    _check(flat_gn[written], flat_pn[written], "cache_nope rows")
    rows_of_slot = np.full(nb * 128, -1)
    rows_of_slot[slots[slots >= 0]] = np.nonzero(slots >= 0)[0]
    _check(flat_gr[written], flat_pr[written], "cache_rope rows", floor[rows_of_slot[written]])


def test_fused_write_bad_slot_flagged_and_skipped():
    T, nb = 64, 2
    v = synth.draw_mla_write(T, nb, 91, device="cuda")
    v["slots"][5] = nb * 128 + 3
    pre = synth.bf16_bits(v["cache_nope"]).reshape(nb * 128, -1)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_rmsnorm_rope_write(v["cache_nope"], v["cache_rope"], v["latent"], v["gamma"], v["cos"],
                               v["sin"], v["slots"], EPS, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 1  # PKV_DEV_BAD_SLOT
    slots = v["slots"].cpu().numpy()
    got = synth.bf16_bits(v["cache_nope"]).reshape(nb * 128, -1)
    untouched = np.ones(nb * 128, dtype=bool)
    untouched[slots[(slots >= 0) & (slots < nb * 128)]] = False
    assert np.array_equal(got[untouched], pre[untouched])


def test_fused_write_full_size_sampled():
    """The bench's size (262,144 tokens): the oracle checks 2,000 sampled tokens."""
    T, nb = 262144, 2048 + 8
    v, pre_n, pre_r, kn, kr = _run(T, nb, 95, outputs=True)
    rng = np.random.default_rng(95)
    rows = np.sort(rng.choice(T, size=2000, replace=False))
    rows = np.unique(np.concatenate([rows, [0, T - 1]]))
    lat = synth.bf16_bits(v["latent"][rows])
    slots = v["slots"].cpu().numpy()[rows]
    sub_n = pre_n.reshape(nb * 128, -1)[slots].reshape(len(rows), 1, 1, 512)
    sub_r = pre_r.reshape(nb * 128, -1)[slots].reshape(len(rows), 1, 1, 64)
    _, _, nope, rope = mw.mla_rmsnorm_rope_write(
        sub_n, sub_r, lat, synth.bf16_bits(v["gamma"]), v["cos"][rows].cpu().numpy(),
        v["sin"][rows].cpu().numpy(), np.full(len(rows), -1, np.int32), 512, EPS)
    _check(synth.bf16_bits(kn[rows]), nope, "k_nope sampled")
    floor = _rope_floor(lat)
    _check(synth.bf16_bits(kr[rows]), rope, "k_rope sampled", floor)
    got_n = synth.bf16_bits(v["cache_nope"]).reshape(nb * 128, -1)[slots]
    got_r = synth.bf16_bits(v["cache_rope"]).reshape(nb * 128, -1)[slots]
    _check(got_n, nope, "cache_nope sampled")
    _check(got_r, rope, "cache_rope sampled", floor)
