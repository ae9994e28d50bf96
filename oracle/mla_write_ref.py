"""Oracle for the fused MLA cache write: RMSNorm of the latent row, RoPE of the rope
row, both written through slot_mapping.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and bench.py's
cpu_baseline / reference leg may import this module; the product library never
does. float64 numpy, written from the pages:

* "昇腾 NPU 独立部署模式 KVCache 自管完整指南", 模式三 (MLA): the fused write takes the
  kv_a projection output (latent 512 + rope 64 per token), the kv_a_layernorm
  weight, cos, sin and slot_mapping, and in one step applies RMSNorm to the latent
  part and RoPE to the rope part and writes nope_cache / rope_cache (optionally
  also returning k_nope / k_rope); "KVCache 优化技能" lists the same operator as the
  fused alternative to the plain scatter write.
* "KV Cache 笔记", the Llama attention forward: RoPE as
  ``x * cos + rotate_half(x) * sin`` with rotate_half(x) = [-x[d/2:], x[:d/2]].

Readings (the pages do not fix them):

* RMSNorm is y = x / sqrt(mean(x^2) + eps) * gamma over the 512 latent values.
* RoPE pairs element i with i + d/2 (the rotate_half form the pages print); cos and
  sin are given per token for all d rope elements.
* Results are rounded to bf16 to nearest, ties to even.
"""
from __future__ import annotations

import numpy as np

from .paged_ref import bf16_bits_to_f64, cache_write


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, round to nearest, ties to even.

    x = m * 2^e with m in [0.5, 1); a bf16 keeps 8 significant bits, so m * 256 is
    rounded to an integer (numpy rounds halves to even) and scaled back. Zeros keep
    their sign. Values must be normal bf16 numbers in range (true for the
    normalised rows and rotated rope values here).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.ldexp(np.round(m * 256.0), e - 8)
    if not np.all(np.isfinite(r)) or np.any((r != 0) & (np.abs(r) < 2.0 ** -126)):
        raise ValueError("value outside the normal bf16 range")
    f32 = r.astype(np.float32)  # exact: r has 8 significant bits
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """Row-wise x / sqrt(mean(x^2) + eps) * gamma (x [T, n], gamma [n])."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gamma


def rope_rotate_half(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """x * cos + rotate_half(x) * sin, rotate_half(x) = [-x[d/2:], x[:d/2]] (x, cos,
    sin [T, d])."""
    h = x.shape[-1] // 2
    rot = np.concatenate([-x[..., h:], x[..., :h]], axis=-1)
    return x * cos + rot * sin


def mla_rmsnorm_rope_write(cache_nope_bits, cache_rope_bits, latent_bits, gamma_bits, cos, sin,
                           slot_mapping, kv_lora_rank: int, eps: float):
    """Returns (cache_nope after, cache_rope after, k_nope bits [T, r], k_rope bits [T, d]).

    latent_bits [T, kv_lora_rank + d] bf16 bits; gamma_bits [kv_lora_rank]; cos, sin
    [T, d] float; caches [nb, bs, 1, width] bf16 bits. Row t of each result goes to
    slot slot_mapping[t] (negative: skipped)."""
    x = bf16_bits_to_f64(latent_bits)
    g = bf16_bits_to_f64(gamma_bits)
    nope = round_to_bf16_bits(rmsnorm(x[:, :kv_lora_rank], g, eps))
    rope = round_to_bf16_bits(rope_rotate_half(x[:, kv_lora_rank:], np.asarray(cos, np.float64),
                                               np.asarray(sin, np.float64)))
    return (cache_write(cache_nope_bits, nope, slot_mapping),
            cache_write(cache_rope_bits, rope, slot_mapping), nope, rope)
