"""Oracle for the quantised KV cache: FP8 E4M3 codes with one fp32 scale per
(token, kv head) row, and attention over the dequantised cache.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and bench.py's
cpu_baseline / reference leg may import this module; the product library never
does. numpy, written from the pages and the format's definition:

* "KVCache 优化技能" (高阶特性): INT8 / W8A8C8 KV cache quantisation;
  "KV Cache 笔记" (Quantized: KIVI-style grouped quantisation, the warning that a
  separate dequantisation per layer and step can eat the bandwidth it saves).
* FP8 E4M3 ("fn" variant of the OCP 8-bit floating point format): 1 sign bit, 4
  exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds subnormals
  m * 2^-9; no infinities; S.1111.111 is NaN; the largest finite value is 448.

Readings (the pages fix no format):

* The group is one (token, kv head) row of head_dim values: scale = amax / 448,
  code = E4M3(x / scale) rounded to nearest even with saturation to +-448; an
  all-zero row has scale 0 and all-zero codes. The scale and the quotient are
  IEEE fp32 divisions, so the library and this oracle take every rounding decision
  on the same fp32 values and the codes are bit-identical.
* Scales are stored per block as [num_blocks, H_kv, block_size] fp32.
* The dequantised value is code * scale; attention is the plain definition over
  the dequantised rows (oracle.paged_ref.paged_decode in float64).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of E4M3 codes (uint8); NaN codes give NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def e4m3_encode(v) -> np.ndarray:
    """E4M3 codes of float values: round to nearest, ties to even, saturating
    finite values to +-448 (the value is rounded first, then clamped)."""
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("NaN input")
    a = np.abs(v)
    # Binade exponent floor(log2 a), exact via frexp (a = f * 2^e, f in [0.5, 1)).
    ex = (np.frexp(np.where(a > 0, a, 1.0))[1] - 1).astype(np.float64)
    ex = np.maximum(ex, -6.0)          # below 2^-6: the subnormal step 2^-9
    q = np.exp2(ex - 3.0)
    r = np.round(a / q) * q           # exact: a / q is a power-of-two scaling
    r = np.minimum(r, E4M3_MAX)
    # Encode the representable magnitude r.
    er = (np.frexp(np.where(r > 0, r, 1.0))[1] - 1).astype(np.float64)
    normal = r >= 2.0 ** -6
    e_field = np.where(normal, er + 7, 0).astype(np.int64)
    m_field = np.where(normal, np.round((r / np.exp2(er) - 1.0) * 8.0), np.round(r / 2.0 ** -9))
    m_field = m_field.astype(np.int64)
    code = (e_field << 3) | m_field
    code = np.where(r == 0, 0, code)
    code = code | np.where(np.signbit(v), 0x80, 0)  # a negative value that rounds to 0 is -0
    return code.astype(np.uint8)


def quantize_rows(x_bits) -> tuple[np.ndarray, np.ndarray]:
    """Rows [..., d] of bf16 bits -> (codes uint8 [..., d], scales float32 [...]).

    scale = amax / 448 and x / scale in IEEE fp32; codes by e4m3_encode."""
    x = (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    v = (x / safe[..., None]).astype(np.float32)
    codes = e4m3_encode(v.astype(np.float64))
    codes = np.where((scale > 0)[..., None], codes, 0).astype(np.uint8)
    return codes, scale


def cache_write_fp8(code_cache, scale_cache, rows_bits, slot_mapping):
    """Quantise rows [T, H_kv, d] (bf16 bits) and store codes at cache
    [nb, bs, H_kv, d][slot] and scales at scale_cache [nb, H_kv, bs][slot // bs, :,
    slot % bs]. Negative slots are skipped. Returns new copies of both."""
    codes, scales = quantize_rows(rows_bits)
    cc = np.array(code_cache, dtype=np.uint8, copy=True)
    sc = np.array(scale_cache, dtype=np.float32, copy=True)
    nb, bs = cc.shape[0], cc.shape[1]
    for t, s in enumerate(np.asarray(slot_mapping).reshape(-1)):
        s = int(s)
        if s < 0:
            continue
        if s >= nb * bs:
            raise IndexError(f"slot {s} outside a cache of {nb * bs} slots")
        cc[s // bs, s % bs] = codes[t]
        sc[s // bs, :, s % bs] = scales[t]
    return cc, sc


def dequantize_cache(code_cache, scale_cache) -> np.ndarray:
    """float64 cache [nb, bs, H_kv, d] = code * scale of its row."""
    vals = e4m3_decode(code_cache)
    s = np.asarray(scale_cache, dtype=np.float64).transpose(0, 2, 1)[..., None]
    return vals * s
