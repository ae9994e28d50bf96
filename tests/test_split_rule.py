"""The attention kernels' softmax rules, restated in float64 and checked
against the oracle's attention (CPU).

The prefill kernel hands the two softmax warps of a query row the two key halves of
every 128-key block (keys [0, 64) and [64, 128)). Each half keeps its own running
maximum in log2 units, raised only when a block's maximum beats it by more than 8, and
rescales its own partial output and normaliser when it does. The halves meet once, at
the end of the row's unit:

    M = max(m_0, m_1),  a_h = 2^(m_h - M)
    o = (a_0 O_0 + a_1 O_1) / (a_0 l_0 + a_1 l_1),  lse = ln 2 * (M + log2(a_0 l_0 + a_1 l_1))

The decode kernels cut a row's keys into split-K pieces at tile boundaries (a CTA's
range of tiles). Each piece runs the same lazy running max over its 128-key tiles and
leaves a normalised partial output and its log2-sum-exp. The merge weighs the pieces by
2^(lse_i - max) (the split merge of the hot path).

The emulations below take those steps in float64 (no bf16 rounding of the weights), so
they must equal softmax attention to rounding for any scores, masks, lengths and cuts.
They check the rules the kernels use, independent of the GPU; the GPU tests compare
the kernels themselves with the oracle.
"""
import math

import numpy as np
import pytest

from oracle import paged_ref as ref

LN2 = math.log(2.0)
BLOCK, HALF = 128, 64


def split_rule(z2, V, rescale=True):
    """z2: one row's scores in log2 units (-inf where masked), V [n, dv]."""
    n, dv = V.shape
    halves = []
    for h in (0, 1):
        m, l, O = -np.inf, 0.0, np.zeros(dv)
        for b0 in range(0, n, BLOCK):
            lo, hi = min(b0 + h * HALF, n), min(b0 + h * HALF + HALF, n)
            zz = z2[lo:hi]
            mt = zz.max() if hi > lo else -np.inf
            if mt > m + 8.0:
                alpha = 0.0 if m == -np.inf else 2.0 ** (m - mt)
                if rescale:
                    O *= alpha
                    l *= alpha
                m = mt
            p = np.zeros(hi - lo) if m == -np.inf else 2.0 ** (zz - m)
            O += p @ V[lo:hi]
            l += p.sum()
        halves.append((m, l, O))
    (m0, l0, O0), (m1, l1, O1) = halves
    M = max(m0, m1)
    a0 = 0.0 if m0 == -np.inf else 2.0 ** (m0 - M)
    a1 = 0.0 if m1 == -np.inf else 2.0 ** (m1 - M)
    lt = a0 * l0 + a1 * l1
    if lt <= 0.0:
        return np.zeros(dv), -np.inf
    return (a0 * O0 + a1 * O1) / lt, LN2 * (M + math.log2(lt))


def _row(rng, n, grow, nvis):
    """Scores (natural units) and values of one row; the first nvis keys are visible
    (a causal prefix). With grow, key block i is scaled by 1 + 1.5 min(i, 8), so later
    blocks beat the running maximum by more than 8 (log2) again and again."""
    z = rng.standard_normal(n) * 3.0
    if grow:
        z *= 1.0 + 1.5 * np.minimum(np.arange(n) // BLOCK, 8)
    visible = np.arange(n) < nvis
    V = rng.standard_normal((n, 16))
    return z, V, visible


CASES = [  # (n, grow, visible prefix)
    (0, False, 0), (1, False, 1), (40, False, 40), (64, False, 64), (65, False, 65),
    (127, True, 127), (128, True, 128), (200, True, 150), (700, True, 700),
    (1000, True, 990), (1500, False, 1200), (513, True, 64), (300, True, 0),
]


@pytest.mark.parametrize("n,grow,nvis", CASES)
def test_split_rule_equals_softmax_attention(n, grow, nvis):
    rng = np.random.default_rng(1000 + n + nvis)
    z, V, visible = _row(rng, max(n, 1), grow, nvis)
    z, V, visible = z[:n], V[:n], visible[:n]
    z2 = np.where(visible, z / LN2, -np.inf)
    o, lse = split_rule(z2, V)
    o_ref, lse_ref, _ = ref.softmax_combine(z, V, visible)
    if nvis == 0:
        assert lse == -np.inf and lse_ref == -np.inf and not o.any()
        return
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12 * max(1.0, np.abs(V).max()))
    assert abs(lse - lse_ref) <= 1e-12 * max(1.0, abs(lse_ref))


def test_growing_rows_do_raise_in_both_halves():
    # The rule's rescale path is exercised: with growing keys each half raises its
    # reference more than once, and the halves end on different references.
    rng = np.random.default_rng(7)
    z, V, visible = _row(rng, 1000, True, 1000)
    z2 = z / LN2
    for h in (0, 1):
        m, raises = -np.inf, 0
        for b0 in range(0, 1000, BLOCK):
            mt = z2[b0 + h * HALF:b0 + h * HALF + HALF].max()
            if mt > m + 8.0:
                raises += m > -np.inf
                m = mt
        assert raises >= 2


def test_dropping_the_rescale_is_caught():
    # A planted mistake in the rule (a raise without rescaling what was accumulated)
    # must move the output away from softmax attention on growing keys.
    rng = np.random.default_rng(8)
    z, V, visible = _row(rng, 1000, True, 1000)
    o_bad, _ = split_rule(z / LN2, V, rescale=False)
    o_ref, _, _ = ref.softmax_combine(z, V, visible)
    assert np.abs(o_bad - o_ref).max() > 1e-3


def piece_rule(z2, V, lo, hi, tile=BLOCK):
    """One split-K piece [lo, hi) of a row as the decode kernels run it: a running max
    over tiles raised only past +8 (log2), rescaling what was accumulated; returns the
    piece's normalised output and log2-sum-exp (the partial the merge reads)."""
    m, l, O = -np.inf, 0.0, np.zeros(V.shape[1])
    for t0 in range(lo, hi, tile):
        zz = z2[t0:min(t0 + tile, hi)]
        mt = zz.max()
        if mt > m + 8.0:
            alpha = 0.0 if m == -np.inf else 2.0 ** (m - mt)
            O *= alpha
            l *= alpha
            m = mt
        p = np.zeros(len(zz)) if m == -np.inf else 2.0 ** (zz - m)
        O += p @ V[t0:t0 + len(zz)]
        l += p.sum()
    if l <= 0.0:
        return np.zeros(V.shape[1]), -np.inf
    return O / l, m + math.log2(l)


def merge_pieces(parts):
    """The log-sum-exp merge of (o_i, lse2_i) pieces: weights 2^(lse2_i - max)."""
    lses = np.array([p[1] for p in parts])
    if np.all(lses == -np.inf):
        return np.zeros_like(parts[0][0]), -np.inf
    mx = lses.max()
    w = np.where(lses == -np.inf, 0.0, 2.0 ** (lses - mx))
    o = sum(wi * p[0] for wi, p in zip(w, parts)) / w.sum()
    return o, LN2 * (mx + math.log2(w.sum()))


@pytest.mark.parametrize("n,cuts", [(1, []), (300, [128]), (1000, [256, 640]), (1000, [128, 256, 384, 896]),
                                    (4097, [1024, 2048, 3072, 4096]), (700, [0, 700])])
def test_split_k_pieces_merged_equal_softmax_attention(n, cuts):
    # Pieces start on tile boundaries (a CTA's range is whole tiles); an empty piece
    # contributes nothing.
    rng = np.random.default_rng(2000 + n + len(cuts))
    z, V, visible = _row(rng, n, True, n)
    z2 = z / LN2
    bounds = [0] + cuts + [n]
    parts = [piece_rule(z2, V, a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    o, lse = merge_pieces(parts)
    o_ref, lse_ref, _ = ref.softmax_combine(z, V, visible)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12 * max(1.0, np.abs(V).max()))
    assert abs(lse - lse_ref) <= 1e-12 * max(1.0, abs(lse_ref))
