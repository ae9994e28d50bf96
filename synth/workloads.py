"""Seeded synthetic workloads for the paged KV cache hot path.

This module only draws inputs: sequence lengths, the initial free-queue order of
the block pool, and N(0,1) values rounded to bf16. It holds none of the
addressing or attention arithmetic; both the oracle and the CUDA path consume
what it draws.

Workload shapes follow the paged-attention problem statement of the pages:
  * physical cache [num_blocks, block_size, H_kv, d_h], block_size 128
    ("model-infer-kvcache" skill note, 模式二 and §3.1);
  * the worked layout batch 2 x max_seq_len 2048 -> 32 blocks, arange table
    (same note, §3.1-3.2);
  * a block pool whose first popped id is the null block
    ("KV Cache 管理设计文档", §2.4 BlockPool);
  * MLA latent cache: kv_lora_rank 512 plus a 64-wide rope key
    (same skill note, 模式三).

Recipe (fixed, stated once): numpy ``default_rng(seed)`` draws the lengths first,
then the pool permutation; torch's generator seeded with ``seed`` draws q, the new
rows and the whole cache in that order, as float32 N(0,1) rounded to bf16 (RNE).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0


@dataclass(frozen=True)
class Workload:
    """One synthetic workload (a batch of sequences over one attention layer)."""

    name: str
    kind: str  # "decode" | "spec_decode" | "mla_decode" | "prefill"
    batch: int
    num_heads: int
    num_kv_heads: int
    head_dim: int  # d_h; for MLA the latent width (kv_lora_rank)
    rope_dim: int = 0  # MLA rope key width
    block_size: int = 128
    scale: float = 0.0
    window: int = 0  # 0 = full attention
    layout: str = "pool"  # "pool" (shuffled BlockPool) or "arange" (static worked layout)
    max_seq_len: int = 0  # arange layout only: tokens per sequence slice
    len_lo: int = 1  # total-length draw bounds (decode) or prior-context bounds (prefill)
    len_hi: int = 1
    q_lo: int = 1  # prefill: new-token count bounds; spec_decode and multi-row MLA
                   # (mla_decode with q_hi > 1): q_lo = q_hi = q_len
    q_hi: int = 1
    forced_q1: int = 0  # prefill: leading sequences forced to q_len 1
    seed: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


def _wl():
    inv = lambda x: 1.0 / float(np.sqrt(x))
    return {
        # Tiny MHA decode on the pages' worked layout (2 x 16 blocks, arange table).
        # The prior kv_len is drawn in [1, 2047] so that the new token at position
        # kv_len stays inside the sequence's 2048-token slice.
        "mha_tiny": Workload(
            name="mha_tiny", kind="decode", batch=2, num_heads=32, num_kv_heads=32,
            head_dim=128, scale=inv(128), layout="arange", max_seq_len=2048,
            len_lo=1, len_hi=2047, seed=1000,
            notes="prior kv_len ~ U[1,2047]; seq_len_kv = kv_len + 1"),
        # GQA decode, long context: the headline workload.
        "gqa_long": Workload(
            name="gqa_long", kind="decode", batch=64, num_heads=64, num_kv_heads=8,
            head_dim=128, scale=inv(128), len_lo=1, len_hi=32768, seed=1001,
            notes="seq_len ~ U[1,32768] incl. the new row; pool = sum(ceil(len/128)) + 1"),
        # Sliding-window GQA decode (window 4096): expired blocks map to the null block.
        "swa": Workload(
            name="swa", kind="decode", batch=32, num_heads=32, num_kv_heads=8,
            head_dim=128, scale=inv(128), window=4096, len_lo=1, len_hi=32768, seed=1002,
            notes="seq_len ~ U[1,32768]; keys at pos < len - 4096 masked"),
        # MLA absorbed decode: key = value = cache_nope (512), plus a 64-wide rope key.
        "mla": Workload(
            name="mla", kind="mla_decode", batch=128, num_heads=128, num_kv_heads=1,
            head_dim=512, rope_dim=64, scale=inv(192), len_lo=1, len_hi=8192, seed=1003,
            notes="seq_len ~ U[1,8192]; scale 1/sqrt(128+64)"),
        # MLA decode of 2 new rows per sequence (the verified token plus one draft,
        # multi-token prediction), bottom-right causal, on the MLA shape above.
        "mla_spec": Workload(
            name="mla_spec", kind="mla_decode", batch=128, num_heads=128, num_kv_heads=1,
            head_dim=512, rope_dim=64, scale=inv(192), len_lo=2, len_hi=8192, q_lo=2, q_hi=2,
            seed=1006, notes="seq_len ~ U[2,8192] incl. the 2 new rows; scale 1/sqrt(128+64)"),
        # Speculative (MTP) decode on the GQA long-context shape: 4 new rows per
        # sequence (the verified token plus 3 drafts), bottom-right causal.
        "spec_decode": Workload(
            name="spec_decode", kind="spec_decode", batch=64, num_heads=64, num_kv_heads=8,
            head_dim=128, scale=inv(128), len_lo=4, len_hi=32768, q_lo=4, q_hi=4, seed=1005,
            notes="seq_len ~ U[4,32768] incl. the 4 new rows"),
        # Mixed chunked prefill + decode batch, causal (bottom-right aligned).
        "mixed_prefill": Workload(
            name="mixed_prefill", kind="prefill", batch=16, num_heads=32, num_kv_heads=8,
            head_dim=128, scale=inv(128), len_lo=0, len_hi=8192, q_lo=1, q_hi=2048,
            forced_q1=4, seed=1004,
            notes="prior ~ U[0,8192], q_len ~ U[1,2048], sequences 0-3 forced to q_len 1"),
    }


WORKLOADS: dict[str, Workload] = _wl()


@dataclass
class Draw:
    """Integer draws of one workload instance (host numpy arrays)."""

    seq_lens: np.ndarray  # int32 [B] total visible length including the new rows
    num_new: np.ndarray  # int32 [B] rows written this step (1 for decode)
    start_pos: np.ndarray  # int32 [B] position of the first new row = seq_lens - num_new
    pool_order: np.ndarray | None  # int32 [num_blocks] initial free-queue order (pool layout)
    num_blocks: int
    max_blocks_per_seq: int


def _ceil_div(a, b):
    return -(-a // b)


def draw(wl: Workload) -> Draw:
    """Draw lengths and the pool's initial free-queue order for ``wl``."""
    rng = np.random.default_rng(wl.seed)
    B, bs = wl.batch, wl.block_size
    if wl.kind == "prefill":
        prior = rng.integers(wl.len_lo, wl.len_hi, size=B, endpoint=True)
        qlen = rng.integers(wl.q_lo, wl.q_hi, size=B, endpoint=True)
        qlen[: wl.forced_q1] = 1
        seq_lens = prior + qlen
        num_new = qlen
    elif wl.kind == "spec_decode" or (wl.kind == "mla_decode" and wl.q_hi > 1):
        seq_lens = rng.integers(wl.len_lo, wl.len_hi, size=B, endpoint=True)
        num_new = np.minimum(seq_lens, wl.q_hi)
    elif wl.layout == "arange":
        kv_len = rng.integers(wl.len_lo, wl.len_hi, size=B, endpoint=True)
        seq_lens = kv_len + 1
        num_new = np.ones(B, dtype=np.int64)
    else:
        seq_lens = rng.integers(wl.len_lo, wl.len_hi, size=B, endpoint=True)
        num_new = np.ones(B, dtype=np.int64)
    seq_lens = seq_lens.astype(np.int32)
    num_new = num_new.astype(np.int32)
    start_pos = (seq_lens - num_new).astype(np.int32)
    if wl.layout == "arange":
        per_seq = wl.max_seq_len // bs
        return Draw(seq_lens, num_new, start_pos, None, B * per_seq, per_seq)
    nblk = _ceil_div(seq_lens.astype(np.int64), bs)
    num_blocks = int(nblk.sum()) + 1  # + the null block
    # The null block is id 0 (first popped); the live ids 1..N-1 are shuffled.
    order = np.concatenate([[0], 1 + rng.permutation(num_blocks - 1)]).astype(np.int32)
    return Draw(seq_lens, num_new, start_pos, order, num_blocks, int(nblk.max()))


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def values(wl: Workload, d: Draw, device="cpu", poison_null: bool = False) -> dict:
    """Draw the bf16 tensors of one instance on ``device``.

    Returns q (and q_rope for MLA), the new rows, and the whole physical cache
    before the write. With ``poison_null`` the null block (id 0 of the pool layout)
    is filled with NaN so that any read of it shows up in the output.
    """
    g = _gen(device, wl.seed)
    B, H, Hkv, dh, bs = wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    T = int(d.num_new.sum())
    out = {}
    if wl.kind == "mla_decode":
        rows = (B, wl.q_hi, H) if wl.q_hi > 1 else (B, H)  # q_hi > 1: q_len rows per sequence
        out["q_nope"] = _randn_bf16(rows + (dh,), g, device)
        out["q_rope"] = _randn_bf16(rows + (wl.rope_dim,), g, device)
        out["nope_new"] = _randn_bf16((T, 1, dh), g, device)
        out["rope_new"] = _randn_bf16((T, 1, wl.rope_dim), g, device)
        out["cache_nope"] = _randn_bf16((d.num_blocks, bs, 1, dh), g, device)
        out["cache_rope"] = _randn_bf16((d.num_blocks, bs, 1, wl.rope_dim), g, device)
        caches = ("cache_nope", "cache_rope")
    else:
        if wl.kind == "spec_decode":
            out["q"] = _randn_bf16((B, wl.q_hi, H, dh), g, device)
        else:
            out["q"] = _randn_bf16((T if wl.kind == "prefill" else B, H, dh), g, device)
        out["k_new"] = _randn_bf16((T, Hkv, dh), g, device)
        out["v_new"] = _randn_bf16((T, Hkv, dh), g, device)
        out["k_cache"] = _randn_bf16((d.num_blocks, bs, Hkv, dh), g, device)
        out["v_cache"] = _randn_bf16((d.num_blocks, bs, Hkv, dh), g, device)
        caches = ("k_cache", "v_cache")
    if poison_null and wl.layout == "pool":
        for c in caches:
            out[c][0].view(torch.int16).fill_(BF16_NAN_BITS)
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit pattern of a tensor as a host uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def draw_explicit(wl: Workload, seq_lens, num_new=None, extra_blocks: int = 0) -> Draw:
    """A Draw with given total lengths (and new-row counts, default 1 per
    non-empty sequence); the pool order is shuffled with ``wl.seed``."""
    rng = np.random.default_rng(wl.seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    if num_new is None:
        num_new = (seq_lens > 0).astype(np.int32)
    num_new = np.asarray(num_new, dtype=np.int32)
    start_pos = (seq_lens - num_new).astype(np.int32)
    nblk = _ceil_div(seq_lens.astype(np.int64), wl.block_size)
    num_blocks = int(nblk.sum()) + 1 + extra_blocks
    order = np.concatenate([[0], 1 + rng.permutation(num_blocks - 1)]).astype(np.int32)
    return Draw(seq_lens, num_new, start_pos, order, num_blocks, max(int(nblk.max()), 1))


def draw_mla_write(num_tokens: int, num_blocks: int, seed: int, device="cpu", block_size: int = 128,
                   rank: int = 512, rope: int = 64, neg_slots: int = 0) -> dict:
    """Inputs of a fused MLA cache write (all drawn here, none computed by the op):

    * latent [T, rank + rope] bf16: N(0,1) rows times a per-row scale exp(U[-2, 2]),
      so the normalisation has work to do;
    * gamma [rank] bf16: 1 + 0.1 N(0,1);
    * cos, sin [T, rope] fp32: the usual RoPE tables of positions ~ U[0, 8192) with
      frequencies 10000^(-2i/rope), i < rope/2, repeated for both halves;
    * slots [T] int32: distinct slots of a [num_blocks, block_size] cache (a random
      permutation), the first ``neg_slots`` replaced by -1;
    * cache_nope [num_blocks, block_size, 1, rank], cache_rope [.., 1, rope] bf16 N(0,1).
    Seeded with numpy default_rng(seed) and a torch generator seeded with seed."""
    rng = np.random.default_rng(seed)
    scale = np.exp(rng.uniform(-2.0, 2.0, size=(num_tokens, 1))).astype(np.float32)
    pos = rng.integers(0, 8192, size=num_tokens).astype(np.float64)
    inv_freq = 10000.0 ** (-np.arange(0, rope, 2, dtype=np.float64) / rope)
    ang = pos[:, None] * inv_freq[None, :]
    ang = np.concatenate([ang, ang], axis=1)
    slots = rng.permutation(num_blocks * block_size)[:num_tokens].astype(np.int32)
    slots[:neg_slots] = -1
    g = _gen(device, seed)
    latent = (torch.randn((num_tokens, rank + rope), generator=g, device=device)
              * torch.from_numpy(scale).to(device)).to(torch.bfloat16)
    gamma = (1.0 + 0.1 * torch.randn((rank,), generator=g, device=device)).to(torch.bfloat16)
    cache_nope = _randn_bf16((num_blocks, block_size, 1, rank), g, device)
    cache_rope = _randn_bf16((num_blocks, block_size, 1, rope), g, device)
    return {
        "latent": latent, "gamma": gamma,
        "cos": torch.from_numpy(np.cos(ang).astype(np.float32)).to(device),
        "sin": torch.from_numpy(np.sin(ang).astype(np.float32)).to(device),
        "slots": torch.from_numpy(slots).to(device),
        "cache_nope": cache_nope, "cache_rope": cache_rope,
    }
