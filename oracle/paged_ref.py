"""fp64 CPU oracle for the paged KV cache write and attention.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and bench.py's
cpu_baseline / reference leg may import this module; the product library never
does, and it shares no code with the CUDA path.

What it computes is the plain definition: paged attention equals attention over
the sequence's keys gathered into contiguous order. Each function names the
passage it follows:

* cache write: a row copy through slot_mapping ("昇腾 NPU 独立部署模式 KVCache
  自管完整指南", 模式二 modeling write: cache.view(-1, H_kv, d)[slot] = row);
* gather: "KVCache 优化技能" §3.1 logical -> physical mapping;
* attention: softmax(q K^T * scale + M) V with the row max subtracted first,
  rows of p summing to one ("KV Cache 笔记", 基线 section "Attention这一格展开"
  and its three engineering details; the decode incremental form after it);
* GQA: query head h reads kv head h // (H / H_kv) (same page, "MHA → MQA → GQA",
  repeat_kv);
* sliding window: the newest W keys are visible (same page, "滑窗与分块"; design
  doc §2.3.2 skip count max(0, n - W + 1));
* causal prefill with a cache offset is bottom-right aligned (same page, sdpa
  section and "手写40行" mask m; standalone guide sparse_mode 3);
* speculative decode: q_len > 1 new rows per sequence under the same bottom-right
  mask (standalone guide appendix C: a multi-token decode step takes the same mask
  branch as prefill);
* MLA absorbed: key = value = cache_nope, and q_rope . cache_rope adds to the
  scores ("KVCache 优化技能" 模式三; standalone guide 模式三; "KV Cache 笔记" MLA),
  for one or several new query rows per sequence (the latter under the same
  bottom-right mask as speculative decode).

All arithmetic is float64; bf16 inputs are widened exactly.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Cache write
# --------------------------------------------------------------------------
def cache_write(cache_bits: np.ndarray, rows_bits: np.ndarray, slot_mapping) -> np.ndarray:
    """Return a copy of ``cache_bits`` [nb, bs, ...] with row t stored at slot[t].

    The cache is viewed as [nb * bs, row] and row t of ``rows_bits`` [T, row...] is
    copied bit for bit to flat index slot_mapping[t]. A negative slot skips the
    row (padding rule of this library, not from the pages); a slot at or past
    nb * bs is an error.
    """
    out = np.array(cache_bits, dtype=np.uint16, copy=True)
    nb, bs = out.shape[0], out.shape[1]
    flat = out.reshape(nb * bs, -1)
    rows = np.asarray(rows_bits, dtype=np.uint16).reshape(len(slot_mapping), flat.shape[1])
    for t, s in enumerate(np.asarray(slot_mapping).reshape(-1)):
        s = int(s)
        if s < 0:
            continue
        if s >= nb * bs:
            raise IndexError(f"slot {s} outside a cache of {nb * bs} slots")
        flat[s] = rows[t]
    return out


# --------------------------------------------------------------------------
# Gather through block_table
# --------------------------------------------------------------------------
def gather_sequence(cache: np.ndarray, table_row, length: int, block_size: int) -> np.ndarray:
    """Contiguous [length, ...] float64 copy of one sequence's rows: row pos comes
    from cache[table_row[pos // bs], pos % bs]. A uint16 cache holds bf16 bit
    patterns and is widened exactly after the gather."""
    out = np.empty((length,) + cache.shape[2:], dtype=cache.dtype)
    for pos in range(length):
        out[pos] = cache[int(table_row[pos // block_size]), pos % block_size]
    return bf16_bits_to_f64(out) if out.dtype == np.uint16 else out.astype(np.float64)


# --------------------------------------------------------------------------
# One query row over a contiguous key set
# --------------------------------------------------------------------------
def softmax_combine(z: np.ndarray, V: np.ndarray, visible: np.ndarray):
    """Softmax over already-scaled scores z [n] (M = 0 where visible, -inf
    elsewhere; the row max is subtracted before exp), then o = p @ V.

    Returns (o [dv], lse, p [n]); lse is the natural-log normaliser
    m + log(sum exp(z - m)). A row with no visible key returns o = 0, lse = -inf.
    """
    if not visible.any():
        return np.zeros(V.shape[1]), -np.inf, np.zeros(len(z))
    z = np.where(visible, z, -np.inf)
    m = z.max()
    e = np.exp(z - m)
    l = e.sum()
    p = e / l
    # o = sum over the visible keys only; masked rows (e.g. expired positions whose
    # table entry is the null block) never enter the sum, whatever they hold.
    return p[visible] @ V[visible], m + np.log(l), p


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, visible: np.ndarray, scale: float):
    """softmax(scale * K q + M) V for one query row; q [dk], K [n, dk], V [n, dv]."""
    return softmax_combine(scale * (K @ q), V, visible)


# --------------------------------------------------------------------------
# Paged decode (one new query token per sequence)
# --------------------------------------------------------------------------
def paged_decode(q, k_cache, v_cache, block_table, seq_lens, block_size: int, scale: float,
                 window: int = 0, batch_indices=None):
    """Decode attention for each (b, h): the query sees positions
    [max(0, len_b - W), len_b) of its sequence (all of [0, len_b) when W = 0).

    q [B, H, d] float64; caches [nb, bs, H_kv, d] float64 or bf16 bits (uint16);
    returns o [B, H, d] and
    lse [B, H] (rows not in ``batch_indices`` stay NaN).
    """
    B, H, _ = q.shape
    Hkv = k_cache.shape[2]
    n_rep = H // Hkv
    o = np.full((B, H, v_cache.shape[3]), np.nan)
    lse = np.full((B, H), np.nan)
    for b in (range(B) if batch_indices is None else batch_indices):
        n = int(seq_lens[b])
        K = gather_sequence(k_cache, block_table[b], n, block_size)
        V = gather_sequence(v_cache, block_table[b], n, block_size)
        pos = np.arange(n)
        visible = pos >= (n - window) if window > 0 else np.ones(n, dtype=bool)
        for h in range(H):
            kv = h // n_rep
            o[b, h], lse[b, h], _ = attend(q[b, h], K[:, kv], V[:, kv], visible, scale)
    return o, lse


# --------------------------------------------------------------------------
# Paged prefill (TND queries, causal bottom-right)
# --------------------------------------------------------------------------
def paged_prefill(q, cu_seqlens_q, k_cache, v_cache, block_table, seq_lens_kv, block_size: int,
                  scale: float, causal: bool = True, rows=None):
    """Prefill attention over TND-packed queries.

    q [T, H, d]; cu_seqlens_q [B] cumulative query ends (no leading zero);
    seq_lens_kv [B] direct total lengths (prior context + new rows). Query row r of
    sequence b (0-based inside the sequence, q_b rows, c_b = len_b - q_b prior
    keys) sees keys j <= c_b + r when causal, all len_b keys otherwise.
    ``rows`` optionally restricts the computed global query rows (others NaN).
    Returns o [T, H, d], lse [T, H].
    """
    T, H, _ = q.shape
    Hkv = k_cache.shape[2]
    n_rep = H // Hkv
    o = np.full((T, H, v_cache.shape[3]), np.nan)
    lse = np.full((T, H), np.nan)
    want = None if rows is None else set(int(r) for r in rows)
    begin = 0
    for b in range(len(cu_seqlens_q)):
        end = int(cu_seqlens_q[b])
        qlen = end - begin
        n = int(seq_lens_kv[b])
        c = n - qlen
        sel = [r for r in range(qlen) if want is None or begin + r in want]
        if sel:
            K = gather_sequence(k_cache, block_table[b], n, block_size)
            V = gather_sequence(v_cache, block_table[b], n, block_size)
            pos = np.arange(n)
            for r in sel:
                visible = pos <= c + r if causal else np.ones(n, dtype=bool)
                for h in range(H):
                    kv = h // n_rep
                    o[begin + r, h], lse[begin + r, h], _ = attend(
                        q[begin + r, h], K[:, kv], V[:, kv], visible, scale)
        begin = end
    return o, lse


# --------------------------------------------------------------------------
# Speculative (multi-token) decode: q_len new rows per sequence, causal
# --------------------------------------------------------------------------
def paged_spec_decode(q, k_cache, v_cache, block_table, seq_lens, block_size: int, scale: float,
                      window: int = 0, batch_indices=None):
    """Decode of q_len new query rows per sequence, all rows already written to the
    cache (MTP / speculative verification; standalone guide, appendix C: q_len > 1
    takes sparse_mode 3, the bottom-right causal mask; design doc, allocate_slots'
    lookahead_tokens reserved for speculative decoding).

    q [B, Q, H, d]; seq_lens [B] total lengths including the Q new rows. Query row
    i of sequence b sits at position len_b - Q + i and sees keys at positions
    p <= len_b - Q + i, and with a window W > 0 only p > len_b - Q + i - W: each row
    is the decode step of the prefix that ends at its own position (reading of the
    pages, which state the window for one query row only). A row whose position is
    negative (len_b < Q) sees no key: o = 0, lse = -inf.
    Returns o [B, Q, H, d] and lse [B, Q, H] (rows not in ``batch_indices`` NaN).
    """
    B, Q, H, _ = q.shape
    Hkv = k_cache.shape[2]
    n_rep = H // Hkv
    o = np.full((B, Q, H, v_cache.shape[3]), np.nan)
    lse = np.full((B, Q, H), np.nan)
    for b in (range(B) if batch_indices is None else batch_indices):
        n = int(seq_lens[b])
        K = gather_sequence(k_cache, block_table[b], n, block_size)
        V = gather_sequence(v_cache, block_table[b], n, block_size)
        pos = np.arange(n)
        for i in range(Q):
            qpos = n - Q + i
            visible = pos <= qpos
            if window > 0:
                visible &= pos > qpos - window
            for h in range(H):
                kv = h // n_rep
                o[b, i, h], lse[b, i, h], _ = attend(q[b, i, h], K[:, kv], V[:, kv], visible, scale)
    return o, lse


# --------------------------------------------------------------------------
# MLA absorbed decode
# --------------------------------------------------------------------------
def mla_decode(q_nope, q_rope, cache_nope, cache_rope, block_table, seq_lens, block_size: int,
               scale: float, batch_indices=None):
    """Absorbed MLA decode: one latent head shared by all H query heads.

    z_j = scale * (q_nope . nope_j + q_rope . rope_j) over positions [0, len_b);
    o = softmax(z) @ nope (key = value = cache_nope). q_nope [B, H, 512],
    q_rope [B, H, 64], cache_nope [nb, bs, 1, 512], cache_rope [nb, bs, 1, 64].
    Returns o [B, H, 512], lse [B, H].
    """
    B, H, dc = q_nope.shape
    o = np.full((B, H, dc), np.nan)
    lse = np.full((B, H), np.nan)
    for b in (range(B) if batch_indices is None else batch_indices):
        n = int(seq_lens[b])
        N = gather_sequence(cache_nope, block_table[b], n, block_size)[:, 0]
        R = gather_sequence(cache_rope, block_table[b], n, block_size)[:, 0]
        visible = np.ones(n, dtype=bool)
        for h in range(H):
            z = scale * (N @ q_nope[b, h] + R @ q_rope[b, h])
            o[b, h], lse[b, h], _ = softmax_combine(z, N, visible)
    return o, lse


def mla_spec_decode(q_nope, q_rope, cache_nope, cache_rope, block_table, seq_lens,
                    block_size: int, scale: float, batch_indices=None):
    """Absorbed MLA decode of Q new query rows per sequence (multi-token prediction
    verification over an MLA cache: standalone guide appendix C, a decode step with
    q_len > 1 takes sparse_mode 3, the bottom-right causal mask; the scores are the
    absorbed ones of 模式三).

    q_nope [B, Q, H, 512], q_rope [B, Q, H, 64]; seq_lens [B] totals including the Q
    new rows. Row i of sequence b sits at position len_b - Q + i and sees the latent
    rows at positions p <= len_b - Q + i. A row whose position is negative
    (len_b < Q) sees none: o = 0, lse = -inf.
    Returns o [B, Q, H, 512] and lse [B, Q, H] (rows not in ``batch_indices`` NaN).
    """
    B, Q, H, dc = q_nope.shape
    o = np.full((B, Q, H, dc), np.nan)
    lse = np.full((B, Q, H), np.nan)
    for b in (range(B) if batch_indices is None else batch_indices):
        n = int(seq_lens[b])
        N = gather_sequence(cache_nope, block_table[b], n, block_size)[:, 0]
        R = gather_sequence(cache_rope, block_table[b], n, block_size)[:, 0]
        pos = np.arange(n)
        for i in range(Q):
            visible = pos <= n - Q + i
            for h in range(H):
                z = scale * (N @ q_nope[b, i, h] + R @ q_rope[b, i, h])
                o[b, i, h], lse[b, i, h], _ = softmax_combine(z, N, visible)
    return o, lse


# --------------------------------------------------------------------------
# Self-checks on a computed row (rows of p sum to one; o is a convex combination)
# --------------------------------------------------------------------------
def check_row(o, p, V, visible) -> None:
    assert abs(p.sum() - 1.0) < 1e-12 or not visible.any()
    if visible.any():
        lo = V[visible].min(axis=0)
        hi = V[visible].max(axis=0)
        assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)
